"""Tensor-core (tcgen05) batched-decode GEMM, batched lm_head and argmax vs the
CPU oracle.  GPU only (marked gpu)."""
import numpy as np
import pytest

import oracle as orc
from gpu_util import assert_close, to_dev, to_host
from w4a16_decode_paged_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    from w4a16_decode_paged_gb300 import api as _api
    from w4a16_decode_paged_gb300 import build
    build.build()
    return _api


@pytest.mark.parametrize("K,N", [(128, 128), (256, 200), (3584, 512), (3584, 4608), (18944, 3584), (896, 130)])
@pytest.mark.parametrize("M", [1, 5, 17, 32])
@pytest.mark.parametrize("split", [False, True])
def test_w4a16_gemm_matches_oracle(api, K, N, M, split):
    r = np.random.default_rng(K * 13 + N + M * 101 + split)
    qw, s = synth.int4_weight(r, N, K)
    x = synth.normal_fp16(r, (M, K))
    bias = synth.normal_fp16(r, (N,), 0.1) if M % 2 else None
    res = synth.normal_fp16(r, (M, N)) if split else None
    ref = orc.w4a16_gemv(x, qw, s, bias=bias, residual=res)
    y = api.w4a16_gemm(to_dev(x, torch), to_dev(qw, torch), to_dev(s, torch),
                       bias=None if bias is None else to_dev(bias, torch),
                       residual=None if res is None else to_dev(res, torch), split=split)
    torch.cuda.synchronize()
    assert_close(to_host(y), ref, what=f"gemm K={K} N={N} M={M} split={split}")


@pytest.mark.parametrize("K,N,M", [(256, 200, 33), (3584, 512, 64), (3584, 512, 128), (896, 130, 100),
                                   (18944, 384, 97)])
@pytest.mark.parametrize("split", [False, True])
def test_w4a16_gemm_wide_row_blocks_match_oracle(api, K, N, M, split):
    """Row blocks wider than a decode batch (a prompt's rows): 64 and 128
    batch columns per weight tile, ragged M and N, K split or not."""
    r = np.random.default_rng(K + 7 * N + 31 * M + split)
    qw, s = synth.int4_weight(r, N, K)
    x = synth.normal_fp16(r, (M, K))
    bias = synth.normal_fp16(r, (N,), 0.1)
    res = synth.normal_fp16(r, (M, N)) if split else None
    ref = orc.w4a16_gemv(x, qw, s, bias=bias, residual=res)
    y = api.w4a16_gemm(to_dev(x, torch), to_dev(qw, torch), to_dev(s, torch), bias=to_dev(bias, torch),
                       residual=None if res is None else to_dev(res, torch), split=split)
    torch.cuda.synchronize()
    assert_close(to_host(y), ref, what=f"wide gemm K={K} N={N} M={M} split={split}")


@pytest.mark.parametrize("K,N,M", [(896, 2432, 64), (3584, 1024, 45)])
def test_w4a16_gemm_silu_mul_wide_row_blocks(api, K, N, M):
    r = np.random.default_rng(K + N + 3 * M)
    qg, sg = synth.int4_weight(r, N, K)
    qu, su = synth.int4_weight(r, N, K)
    x = synth.normal_fp16(r, (M, K))
    ref = orc.silu_mul(orc.w4a16_gemv(x, qg, sg), orc.w4a16_gemv(x, qu, su))
    y = api.w4a16_gemm_silu_mul(to_dev(x, torch), to_dev(qg, torch), to_dev(sg, torch), to_dev(qu, torch),
                                to_dev(su, torch))
    torch.cuda.synchronize()
    assert_close(to_host(y), ref, what=f"wide gemm silu K={K} N={N} M={M}")


def test_w4a16_gemm_rejects_rows_beyond_the_widest_block(api):
    r = np.random.default_rng(4)
    qw, s = synth.int4_weight(r, 128, 256)
    with pytest.raises(Exception):
        api.w4a16_gemm(to_dev(synth.normal_fp16(r, (129, 256)), torch), to_dev(qw, torch), to_dev(s, torch))
    with pytest.raises(Exception):
        api.w4a16_gemm_silu_mul(to_dev(synth.normal_fp16(r, (65, 256)), torch), to_dev(qw, torch), to_dev(s, torch),
                                to_dev(qw, torch), to_dev(s, torch))


def test_w4a16_gemm_repeat_calls_leave_counters_zero(api):
    r = np.random.default_rng(3)
    qw, s = synth.int4_weight(r, 3584, 18944)
    x = to_dev(synth.normal_fp16(r, (32, 18944)), torch)
    qd, sd = to_dev(qw, torch), to_dev(s, torch)
    ws = torch.zeros(api.load().w4a16_gemm_workspace_size(32, 18944, 3584, 0), dtype=torch.uint8, device="cuda")
    y1 = api.w4a16_gemm(x, qd, sd, workspace=ws)
    y2 = api.w4a16_gemm(x, qd, sd, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_one_workspace_serves_projections_of_different_shapes(api):
    """The decoder layer's four projections in turn on one split-K workspace
    (its tickets sit at a fixed place whatever the shape), twice over."""
    r = np.random.default_rng(11)
    M = 32
    shapes = [(3584, 4608, False), (3584, 3584, False), (3584, 18944, True), (18944, 3584, False)]
    lib = api.load()
    ws = torch.zeros(max(lib.w4a16_gemm_workspace_size(M, K, N, int(silu)) for K, N, silu in shapes),
                     dtype=torch.uint8, device="cuda")
    cases = []
    for K, N, silu in shapes:
        x = synth.normal_fp16(r, (M, K))
        w = [synth.int4_weight(r, N, K) for _ in range(2 if silu else 1)]
        if silu:
            ref = orc.silu_mul(orc.w4a16_gemv(x, *w[0]), orc.w4a16_gemv(x, *w[1]))
        else:
            ref = orc.w4a16_gemv(x, *w[0])
        cases.append((to_dev(x, torch), [(to_dev(q, torch), to_dev(s_, torch)) for q, s_ in w], silu, ref))
    for rep in range(2):
        outs = []
        for x, w, silu, ref in cases:
            if silu:
                outs.append(api.w4a16_gemm_silu_mul(x, w[0][0], w[0][1], w[1][0], w[1][1], workspace=ws))
            else:
                outs.append(api.w4a16_gemm(x, w[0][0], w[0][1], workspace=ws))
        torch.cuda.synchronize()
        for y, (_, _, _, ref) in zip(outs, cases):
            assert_close(to_host(y), ref, what=f"shared workspace pass {rep}")


@pytest.mark.parametrize("K,N,M", [(896, 2432, 32), (3584, 18944, 32), (3584, 256, 9)])
def test_w4a16_gemm_silu_mul_matches_oracle(api, K, N, M):
    r = np.random.default_rng(K + N + M)
    qg, sg = synth.int4_weight(r, N, K)
    qu, su = synth.int4_weight(r, N, K)
    x = synth.normal_fp16(r, (M, K))
    ref = orc.silu_mul(orc.w4a16_gemv(x, qg, sg), orc.w4a16_gemv(x, qu, su))
    y = api.w4a16_gemm_silu_mul(to_dev(x, torch), to_dev(qg, torch), to_dev(sg, torch), to_dev(qu, torch),
                                to_dev(su, torch))
    torch.cuda.synchronize()
    assert_close(to_host(y), ref, what="gemm silu")


def test_w4a16_gemv_routes_batches_to_tensor_cores(api):
    r = np.random.default_rng(8)
    qw, s = synth.int4_weight(r, 512, 3584)
    x = synth.normal_fp16(r, (8, 3584))
    y = api.w4a16_gemv(to_dev(x, torch), to_dev(qw, torch), to_dev(s, torch))
    torch.cuda.synchronize()
    assert_close(to_host(y), orc.w4a16_gemv(x, qw, s), what="gemv M=8")


@pytest.mark.parametrize("B,H,V", [(32, 3584, 152064), (5, 896, 1000)])
def test_batched_lm_head_and_argmax(api, B, H, V):
    r = np.random.default_rng(B * V)
    W = synth.normal_fp16(r, (V, H), std=0.02)
    x = synth.normal_fp16(r, (B, H))
    lg = api.lm_head_logits_batched(to_dev(x, torch), to_dev(W, torch))
    l16 = torch.empty((B, V), dtype=torch.float16, device="cuda")
    toks = api.argmax_rows(lg, logits16=l16)
    torch.cuda.synchronize()
    lg, toks = to_host(lg), to_host(toks)
    for b in range(0, B, max(1, B // 4)):
        ref = orc.fp16_gemv(x[b], W)
        assert_close(lg[b], ref, atol=1e-3, rtol=1e-4, what="lm_head fp32 logits")
        srt = np.sort(ref)
        if srt[-1] - srt[-2] > 1e-3:
            assert toks[b] == orc.argmax(ref)
    assert np.array_equal(to_host(l16), lg.astype(np.float16))


def test_argmax_rows_ties_lowest_index(api):
    lg = torch.zeros((2, 5000), dtype=torch.float32, device="cuda")
    lg[0, 4000] = 3.0
    lg[0, 17] = 3.0
    lg[1, :] = -1.0
    toks = api.argmax_rows(lg)
    torch.cuda.synchronize()
    assert to_host(toks).tolist() == [17, 0]


@pytest.mark.parametrize("B,V", [(33, 152064), (3, 1001), (2, 7), (1, 8)])
def test_argmax_rows_slices_ties_nan(api, B, V):
    """Row argmax over slices of the row: random rows, a tie planted across
    two slices (the lower index wins), a row with NaN entries (skipped), a
    row of NaN only (-1), negative rows; fp16 copy of the logits."""
    r = np.random.default_rng(7000 + V)
    lg = r.standard_normal((B, V)).astype(np.float32)
    if V >= 16:
        i0, i1 = V // 8 + 1, V - 2              # different slices of eight
        lg[0, i1] = lg[0, i0] = lg[0].max() + 1.0
    if B >= 3:
        lg[1, ::3] = np.nan
        lg[2, :] = -np.abs(lg[2, :]) - 1.0
    if B >= 2 and V < 16:
        lg[1, :] = np.nan
    d = to_dev(lg, torch)
    l16 = torch.empty((B, V), dtype=torch.float16, device="cuda")
    toks = to_host(api.argmax_rows(d, logits16=l16)).tolist()
    torch.cuda.synchronize()
    for b in range(B):
        row = lg[b]
        want = -1 if np.all(np.isnan(row)) else int(np.nanargmax(row))
        assert toks[b] == want, (b, toks[b], want)
    got16 = to_host(l16)
    assert np.array_equal(np.isnan(got16), np.isnan(lg))
    m = ~np.isnan(lg)
    assert np.array_equal(got16[m], lg[m].astype(np.float16))
