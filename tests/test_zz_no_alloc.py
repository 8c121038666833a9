"""paged_gqa_decode_noalloc: the allocation-free attention entry point.

Some callers cannot allocate device memory (a plugin that only receives
input/output pointers from a host framework owning the memory pool, or code
running inside a global-mode stream capture where cudaMalloc is illegal).
For them the split-K scratch lives in a static device array inside the
library.  This file runs last so that a failure here leaves every other test
already run.  GPU only (marked gpu)."""
import math

import numpy as np
import pytest

import oracle as orc
from gpu_util import assert_close, to_dev, to_host
from w4a16_decode_paged_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from w4a16_decode_paged_gb300 import _lib, build
    build.build()
    orc.build()
    return _lib.load()


def _host_case(seed, lens, Hq=28, Hkv=4, D=128):
    r = np.random.default_rng(seed)
    pages = int(sum((L + 15) // 16 for L in lens)) + 9
    kp = synth.kv_pool(r, pages, Hkv, D)
    vp = synth.kv_pool(r, pages, Hkv, D)
    bt = synth.block_table(r, lens, pages)
    q = synth.normal_fp16(r, (len(lens), Hq, D), std=2.0)
    return q, kp, vp, bt, np.asarray(lens, np.int32)


def _case(seed, lens, Hq=28, Hkv=4, D=128):
    return [to_dev(a, torch) for a in _host_case(seed, lens, Hq, Hkv, D)]


def _run(lib, fn, q, kp, vp, bt, ln, max_context, part, ws=None):
    B, Hq, D = q.shape
    Hkv = kp.shape[1]
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream().cuda_stream
    args = [q.data_ptr(), 0, kp.data_ptr(), vp.data_ptr(), kp.shape[0], bt.data_ptr(), bt.shape[1], ln.data_ptr(),
            max_context, B, Hq, Hkv, D, 1.0 / math.sqrt(D), part]
    if fn == "paged_gqa_decode":
        rc = lib.paged_gqa_decode(*args, ws.data_ptr(), ws.numel(), out.data_ptr(), None, stream)
    else:
        rc = lib.paged_gqa_decode_noalloc(*args, out.data_ptr(), None, stream)
    assert rc == 0, lib.w4a16_last_error()
    return out


def test_noalloc_matches_workspace_version_two_calls_in_a_row(lib):
    lens = [1, 17, 513, 2000]
    part, max_context = 64, 2000
    B, Hq, Hkv = len(lens), 28, 4
    ws = torch.zeros(lib.paged_gqa_decode_workspace_size(B, Hq, Hkv, max_context, part, 128), dtype=torch.uint8,
                     device="cuda")
    assert ws.numel() <= 4 << 20  # fits the static scratch
    for seed in (1, 2):  # second call with new data: nothing may leak from the first
        q, kp, vp, bt, ln = _case(seed, lens)
        ref = _run(lib, "paged_gqa_decode", q, kp, vp, bt, ln, max_context, part, ws)
        got = _run(lib, "paged_gqa_decode_noalloc", q, kp, vp, bt, ln, max_context, part)
        torch.cuda.synchronize()
        assert_close(to_host(got), to_host(ref), what=f"noalloc call {seed}")


def test_noalloc_matches_oracle_across_partitions(lib):
    """The static-scratch path against the CPU oracle directly: lengths on
    both sides of a page and of a 64-token partition, so the partials of
    several partitions meet in the static array's merge."""
    lens = [1, 15, 16, 17, 63, 64, 65, 700]
    part, max_context = 64, 700
    hq, hkp, hvp, hbt, hln = _host_case(11, lens)
    q, kp, vp, bt, ln = (to_dev(a, torch) for a in (hq, hkp, hvp, hbt, hln))
    got = _run(lib, "paged_gqa_decode_noalloc", q, kp, vp, bt, ln, max_context, part)
    torch.cuda.synchronize()
    ref = orc.paged_attention(hq, hkp, hvp, hbt, hln, 1.0 / math.sqrt(hq.shape[2]))
    assert_close(to_host(got), ref, what="noalloc vs oracle")


def test_noalloc_rejects_sizes_beyond_the_static_scratch(lib):
    q, kp, vp, bt, ln = _case(3, [40])
    out = torch.empty_like(q)
    # 64 sequences x 28 heads x 64 partitions of partials is far beyond 4 MiB
    rc = lib.paged_gqa_decode_noalloc(q.data_ptr(), 0, kp.data_ptr(), vp.data_ptr(), kp.shape[0], bt.data_ptr(), 2048,
                                      ln.data_ptr(), 32768, 64, 28, 4, 128, 0.088, 512, out.data_ptr(), None,
                                      torch.cuda.current_stream().cuda_stream)
    assert rc == 3 and b"static array holds" in lib.w4a16_last_error()
