"""bench.py's continuous-batching measurement on the GPU, over a 2-layer
model of the small test shapes: the real scheduler reproduces the loop's
accounting (p + n - 1 steps per sequence, n tokens out, no preemption when
every slot has room for its longest sequence, every page back at the end).
Runs last (file name): it only adds the bench mode's own check to the
kernel and scheduler tests before it."""
import os
import sys
import time

import numpy as np
import pytest

from gpu_util import to_dev
from w4a16_decode_paged_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_bench_batching_mode_on_a_small_model():
    from w4a16_decode_paged_gb300 import api, build
    build.build()
    cfg = dict(synth.TINY_LAYER, n_layers=2, vocab=600, bias=True, codes="symmetric")
    r = synth.rng(8200)
    layers = [synth.layer_weights(r, cfg) for _ in range(2)]
    embed = to_dev(synth.normal_fp16(r, (cfg["vocab"], cfg["hidden"])), torch)
    fnorm = to_dev(synth.gamma(r, cfg["hidden"]), torch)
    lm = to_dev(synth.normal_fp16(r, (cfg["vocab"], cfg["hidden"]), std=0.02), torch)
    Hkv, D = cfg["n_kv_heads"], cfg["head_dim"]
    zeros = lambda n: (torch.zeros((n, Hkv, 16, D), dtype=torch.float16, device="cuda"),
                       torch.zeros((n, Hkv, 16, D), dtype=torch.float16, device="cuda"))
    res = bench.time_batching(api, cfg, layers, embed, fnorm, lm, zeros, torch.cuda.synchronize, time.perf_counter,
                              n_seq=6, max_batch=4, new_tokens=4, seed=11)
    plens = bench.batching_prompts(11, 6)
    assert res["generated_tokens"] == 6 * 4
    assert res["token_steps"] == sum(p + 4 - 1 for p in plens)
    assert res["preemptions"] == 0
    assert res["free_pages_after"] == res["num_pages"]
    assert 1.0 <= res["mean_batch"] <= 4.0 and res["seconds"] > 0
    assert np.isfinite(res["generated_tok_per_s"])
