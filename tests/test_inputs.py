"""The seeded input recipe and the benchmark's byte counts (CPU).

The inputs must have the structure the decode path assumes (disjoint pages
per sequence, -1 past each sequence's last page, the forced 15/16/17 page
boundary lengths, the int4 code distributions), and the roofline
denominator in bench.py must equal the bytes of the arrays a step really
reads and writes."""
import math

import numpy as np
import pytest

from w4a16_decode_paged_gb300 import synth

PAGE = 16


def _nibbles(qw):
    w = qw.astype(np.uint64)
    return np.stack([(w >> (4 * i)) & 0xF for i in range(8)], axis=-1)


def test_qwen_shapes_are_gqa_7_to_1():
    for cfg in (synth.QWEN_LAYER, synth.QWEN_MODEL, synth.QWEN_BATCHED, synth.QWEN_LONG):
        assert (cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["inter"]) == \
            (3584, 28, 4, 128, 18944)
        assert cfg["n_q_heads"] // cfg["n_kv_heads"] == 7
    assert synth.QWEN_MODEL["n_layers"] == synth.QWEN_BATCHED["n_layers"] == 28
    assert synth.QWEN_MODEL["vocab"] == synth.QWEN_BATCHED["vocab"] == 152064


def test_block_table_pages_are_disjoint_and_cover_each_sequence():
    r = synth.rng(5)
    lens = np.array([1, 15, 16, 17, 31, 32, 33, 0, 4096], np.int32)
    pool = 400
    bt = synth.block_table(r, lens, pool)
    seen = set()
    for b, L in enumerate(lens):
        need = (int(L) + PAGE - 1) // PAGE
        row = bt[b]
        assert np.all((row[:need] >= 0) & (row[:need] < pool))
        assert np.all(row[need:] == -1)
        assert not seen & set(row[:need].tolist())
        seen |= set(row[:need].tolist())
    assert len(seen) == sum((int(L) + PAGE - 1) // PAGE for L in lens)
    with pytest.raises(AssertionError):
        synth.block_table(r, [PAGE * 10 + 1], 10)


def test_batched_lengths_force_the_page_boundaries():
    cfg = synth.QWEN_BATCHED
    lens = synth.batched_lens(synth.rng(cfg["seed"]), cfg["batch"], cfg["max_context"], cfg["forced_lens"])
    assert list(lens[:3]) == [15, 16, 17]
    assert lens.min() >= 1 and lens.max() <= cfg["max_context"] and len(lens) == 32


def test_int4_code_distributions():
    r = synth.rng(6)
    qw, s = synth.int4_weight(r, 64, 1024, "full")
    assert qw.dtype == np.uint32 and qw.shape == (64, 128) and s.shape == (64, 8) and s.dtype == np.float16
    counts = np.bincount(_nibbles(qw).ravel().astype(np.int64), minlength=16)
    assert np.all(counts > 0.8 * counts.mean())          # every code of [-8, 7] about equally often
    assert s.min() >= np.float16(0.005) and s.max() <= np.float16(0.02)
    qs, _ = synth.int4_weight(r, 64, 1024, "symmetric")
    u = _nibbles(qs).ravel().astype(np.int64)
    assert np.all(u != 0)                                 # no code -8 (offset binary 0)
    counts = np.bincount(u, minlength=16)[1:]
    assert np.all(counts > 0.8 * counts.mean())          # codes -7..7 about equally often
    assert abs(float(np.mean(u - 8))) < 0.02


def test_model_case_pools_hold_data_only_on_named_pages():
    cfg = dict(synth.TINY_LAYER, n_layers=2, vocab=50, seed=9)
    case = synth.model_case(cfg, lens=[0, 17, 33], gen_tokens=4, pool_pages=20)
    bt = case["bt"]
    named = np.unique(bt[bt >= 0])
    assert np.array_equal(case["used_pages"], named)
    assert bt.shape[1] == (33 + 4 + PAGE - 1) // PAGE
    for layer in range(2):
        for which in "kv":
            p = synth.host_pool(case, layer, which)
            assert p.shape == (20, cfg["n_kv_heads"], PAGE, cfg["head_dim"])
            idle = np.setdiff1d(np.arange(20), named)
            assert not p[idle].any()
            assert np.all(np.abs(p[named]).sum(axis=(1, 2, 3)) > 0)
    assert case["tok"].min() >= 0 and case["tok"].max() < 50


def test_same_seed_same_inputs():
    a = synth.model_case(dict(synth.TINY_LAYER, vocab=10), lens=[5])
    b = synth.model_case(dict(synth.TINY_LAYER, vocab=10), lens=[5])
    assert np.array_equal(a["layers"][0]["wq"], b["layers"][0]["wq"])
    assert np.array_equal(a["k_used"][0], b["k_used"][0]) and np.array_equal(a["tok"], b["tok"])


def test_bench_bytes_equal_the_arrays_a_step_touches():
    """bench.layer_bytes / step_bytes against the nbytes of the arrays one
    b=1 step reads and writes: every int4 weight, scale and bias array of a
    layer, the activations in and out of each projection (gate|up writes I
    values, not 2I), the K/V rows of the cached tokens, the page table, q and
    the attention output; then 28 layers plus the lm_head matrix and the
    hidden state."""
    import bench
    cfg = synth.QWEN_MODEL
    w = synth.layer_weights(synth.rng(1), dict(cfg, codes="full"))
    weights = sum(w[k].nbytes for k in w if k[0] in "wsb" and w[k] is not None)
    H, Hq, Hkv, D, I = 3584, 28, 4, 128, 18944
    act = 2 * ((H + (Hq + 2 * Hkv) * D) + (Hq * D + 2 * H) + (H + I) + (I + 2 * H))
    L = 513
    kv = 2 * Hkv * L * D * 2
    att = kv + 4 * math.ceil(L / PAGE) + 2 * Hq * D * 2
    g, a = bench.layer_bytes(cfg, [L])
    assert g == weights + act
    assert a == att
    assert bench.step_bytes(cfg, [L]) == 28 * (weights + act + att) + cfg["vocab"] * H * 2 + H * 2
    # the b=1 figure quoted with the roofline: about 4.49 GB per token
    assert abs(bench.step_bytes(cfg, [L]) / 1e9 - 4.49) < 0.01


def test_clock_sampler_reads_samples_from_the_pipe():
    """bench.ClockSampler against a stand-in for nvidia-smi that prints two
    kinds of CSV samples: median SM clock, max clock and the active throttle
    reasons, from the lines read off its stdout."""
    import time

    import bench
    line_a = "0, 2070, 2070, 812.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active"
    line_b = "0, 1980, 2070, 990.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"
    script = f'while true; do echo "{line_a}"; echo "{line_b}"; echo "{line_a}"; sleep 0.05; done'
    with bench.ClockSampler(0, command=["sh", "-c", script]) as clk:
        time.sleep(0.3)
    s = clk.summary()
    assert s["samples"] >= 3 and s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert clk.lines[0] == line_a


def test_clock_sampler_without_nvidia_smi():
    import bench
    with bench.ClockSampler(0, command=["/nonexistent/nvidia-smi"]) as clk:
        pass
    assert clk.summary()["reasons"] == ["unavailable"]
