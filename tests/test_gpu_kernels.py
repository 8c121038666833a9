"""Parity of each C-ABI kernel call with the CPU oracle on seeded inputs.
GPU only (marked gpu)."""
import math

import numpy as np
import pytest

import oracle as orc
from gpu_util import assert_close, max_rel, to_dev, to_host
from w4a16_decode_paged_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    from w4a16_decode_paged_gb300 import api as _api
    from w4a16_decode_paged_gb300 import build
    build.build()
    return _api


# ----------------------------------------------------------------------------- GEMV

GEMV_SHAPES = [(128, 1), (256, 37), (896, 128), (896, 1152), (896, 2432), (2432, 896), (1024, 64),
               (3584, 130), (3584, 131), (3584, 2), (3584, 6), (3584, 512), (3584, 4608), (3584, 18944),
               (18944, 3584), (18944, 14)]


@pytest.mark.parametrize("K,N", GEMV_SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_w4a16_gemv_matches_oracle(api, K, N, M):
    r = np.random.default_rng(K * 31 + N * 7 + M)
    qw, s = synth.int4_weight(r, N, K)
    x = synth.normal_fp16(r, (M, K))
    bias = synth.normal_fp16(r, (N,), 0.1) if (N + M) % 2 == 0 else None
    res = synth.normal_fp16(r, (M, N)) if M % 2 == 1 else None
    ref = orc.w4a16_gemv(x, qw, s, bias=bias, residual=res)
    y = api.w4a16_gemv(to_dev(x, torch), to_dev(qw, torch), to_dev(s, torch),
                       bias=None if bias is None else to_dev(bias, torch),
                       residual=None if res is None else to_dev(res, torch))
    torch.cuda.synchronize()
    assert_close(to_host(y), ref, what=f"gemv K={K} N={N} M={M}")


@pytest.mark.parametrize("K,N,M", [(896, 1152, 1), (3584, 4608, 1), (3584, 4608, 2), (896, 37, 3),
                                   (18944, 130, 3), (18944, 3584, 4)])
def test_w4a16_gemv_rmsnorm_matches_oracle(api, K, N, M):
    r = np.random.default_rng(K + N + 5 * M)
    qw, s = synth.int4_weight(r, N, K)
    x = synth.normal_fp16(r, (M, K), std=3.0)
    g = synth.gamma(r, K)
    bias = synth.normal_fp16(r, (N,), 0.1)
    ref = orc.w4a16_gemv(orc.rmsnorm(x, g, 1e-6), qw, s, bias=bias)
    y = api.w4a16_gemv_rmsnorm(to_dev(x, torch), to_dev(g, torch), 1e-6, to_dev(qw, torch), to_dev(s, torch),
                               bias=to_dev(bias, torch))
    torch.cuda.synchronize()
    assert_close(to_host(y), ref, what="gemv_rmsnorm")


@pytest.mark.parametrize("K,N,M,norm", [(896, 2432, 1, True), (3584, 18944, 1, True), (3584, 18944, 2, False),
                                        (256, 40, 4, True), (3584, 10, 1, True), (3584, 7, 3, False),
                                        (18944, 10, 3, True), (18944, 64, 4, False)])
def test_w4a16_gemv_silu_mul_matches_oracle(api, K, N, M, norm):
    r = np.random.default_rng(K * 3 + N + M)
    qg, sg = synth.int4_weight(r, N, K)
    qu, su = synth.int4_weight(r, N, K)
    x = synth.normal_fp16(r, (M, K))
    g = synth.gamma(r, K) if norm else None
    xn = orc.rmsnorm(x, g, 1e-6) if norm else x
    ref = orc.silu_mul(orc.w4a16_gemv(xn, qg, sg), orc.w4a16_gemv(xn, qu, su))
    y = api.w4a16_gemv_silu_mul(to_dev(x, torch), None if g is None else to_dev(g, torch), 1e-6,
                                to_dev(qg, torch), to_dev(sg, torch), to_dev(qu, torch), to_dev(su, torch))
    torch.cuda.synchronize()
    assert_close(to_host(y), ref, what="gemv_silu_mul")


def test_gemv_is_deterministic_and_leaves_inputs(api):
    r = np.random.default_rng(77)
    qw, s = synth.int4_weight(r, 3584, 3584)
    x = synth.normal_fp16(r, (1, 3584))
    xd, qd, sd = to_dev(x, torch), to_dev(qw, torch), to_dev(s, torch)
    y1 = api.w4a16_gemv(xd, qd, sd)
    y2 = api.w4a16_gemv(xd, qd, sd)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert np.array_equal(to_host(xd), x) and np.array_equal(to_host(qd).view(np.uint32), qw)


# ----------------------------------------------------------------------------- RMSNorm

@pytest.mark.parametrize("M,H", [(1, 896), (3, 3584), (2, 18944), (1, 8)])
def test_rmsnorm_matches_oracle(api, M, H):
    r = np.random.default_rng(M * H)
    x = synth.normal_fp16(r, (M, H), std=2.0)
    g = synth.gamma(r, H)
    ref = orc.rmsnorm(x, g, 1e-6)
    y = api.rmsnorm(to_dev(x, torch), to_dev(g, torch), 1e-6)
    torch.cuda.synchronize()
    assert_close(to_host(y), ref, what="rmsnorm")


# ----------------------------------------------------------------------------- RoPE + append

@pytest.mark.parametrize("Hq,Hkv", [(7, 1), (28, 4)])
@pytest.mark.parametrize("fused", [False, True])
def test_kv_append_rope_placement_bit_exact(api, Hq, Hkv, fused):
    r = np.random.default_rng(Hq * 10 + int(fused))
    D, theta = 128, 1e6
    lens = np.array([1, 15, 16, 17, 31, 32, 33, 37], np.int32)
    B = len(lens)
    pages = int(sum((L + 15) // 16 for L in lens)) + 5
    kp = synth.kv_pool(r, pages, Hkv, D)
    vp = synth.kv_pool(r, pages, Hkv, D)
    bt = synth.block_table(r, lens, pages, max_blocks=4)
    q = synth.normal_fp16(r, (B, Hq, D))
    k = synth.normal_fp16(r, (B, Hkv, D))
    v = synth.normal_fp16(r, (B, Hkv, D))
    q_ref = np.stack([orc.rope(q[b], int(lens[b]) - 1, theta) for b in range(B)])
    k_rot = np.stack([orc.rope(k[b], int(lens[b]) - 1, theta) for b in range(B)])
    kp_ref, vp_ref = kp.copy(), vp.copy()
    orc.kv_append(k_rot, v, kp_ref, vp_ref, bt, lens)

    kpd, vpd = to_dev(kp, torch), to_dev(vp, torch)
    if fused:  # q|k|v rows of one buffer, as the decode step lays them out
        row = np.concatenate([q.reshape(B, -1), k.reshape(B, -1), v.reshape(B, -1)], axis=1)
        rd = to_dev(row, torch)
        qd = rd[:, :Hq * D]
        kd = rd[:, Hq * D:(Hq + Hkv) * D]
        vd = rd[:, (Hq + Hkv) * D:]
        from w4a16_decode_paged_gb300._lib import check, load
        btd, ld = to_dev(bt, torch), to_dev(lens, torch)  # kept alive until the launch is enqueued
        check(load().kv_append_rope(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), row.shape[1], kpd.data_ptr(),
                                    vpd.data_ptr(), pages, btd.data_ptr(), bt.shape[1], ld.data_ptr(), B, Hq,
                                    Hkv, D, theta, None, torch.cuda.current_stream().cuda_stream))
        torch.cuda.synchronize()
        q_got = to_host(rd)[:, :Hq * D].reshape(B, Hq, D)
    else:
        qd = to_dev(q, torch)
        btd, ld = to_dev(bt, torch), to_dev(lens, torch)
        api.kv_append_rope(qd, to_dev(k, torch), to_dev(v, torch), kpd, vpd, btd, ld, theta)
        torch.cuda.synchronize()
        q_got = to_host(qd)
    assert_close(q_got, q_ref, what="rope q")
    kp_got, vp_got = to_host(kpd), to_host(vpd)
    # exactly the appended slots changed
    expect = {(int(bt[b, (lens[b] - 1) // 16]), h, int((lens[b] - 1) % 16)) for b in range(B) for h in range(Hkv)}
    changed_v = {tuple(int(i) for i in t) for t in np.argwhere(np.any(vp_got != vp, axis=-1))}
    assert changed_v <= expect
    assert np.array_equal(vp_got, vp_ref)  # v placement and values bit-exact
    mask = np.zeros(kp.shape[:3], bool)
    for (pg, h, sl) in expect:
        mask[pg, h, sl] = True
    assert np.array_equal(kp_got[~mask], kp[~mask])  # nothing else in the K pool moved
    assert_close(kp_got[mask], kp_ref[mask], what="rope k in pool")


def test_kv_append_rope_long_position_angles(api):
    r = np.random.default_rng(5)
    D, Hq, Hkv, theta = 128, 28, 4, 1e6
    lens = np.array([32768, 513], np.int32)
    bt = np.full((2, 2048), -1, np.int32)
    bt[0, 2047] = 3
    bt[1, 32] = 1
    kp = synth.kv_pool(r, 4, Hkv, D)
    vp = synth.kv_pool(r, 4, Hkv, D)
    q = synth.normal_fp16(r, (2, Hq, D))
    k = synth.normal_fp16(r, (2, Hkv, D))
    v = synth.normal_fp16(r, (2, Hkv, D))
    qd, kpd, vpd = to_dev(q, torch), to_dev(kp, torch), to_dev(vp, torch)
    api.kv_append_rope(qd, to_dev(k, torch), to_dev(v, torch), kpd, vpd, to_dev(bt, torch), to_dev(lens, torch),
                       theta)
    torch.cuda.synchronize()
    for b in range(2):
        assert_close(to_host(qd)[b], orc.rope(q[b], int(lens[b]) - 1, theta), what="rope q long")
        pg, sl = int(bt[b, (lens[b] - 1) // 16]), int((lens[b] - 1) % 16)
        assert_close(to_host(kpd)[pg, :, sl], orc.rope(k[b], int(lens[b]) - 1, theta), what="rope k long")


def test_kv_append_rope_bad_page_sets_flag(api):
    r = np.random.default_rng(6)
    kp = synth.kv_pool(r, 4, 1, 128)
    vp = kp.copy()
    bt = np.array([[0, 99]], np.int32)  # second page out of range
    lens = np.array([20], np.int32)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    kpd, vpd = to_dev(kp, torch), to_dev(vp, torch)
    q = to_dev(synth.normal_fp16(r, (1, 7, 128)), torch)
    kv = to_dev(synth.normal_fp16(r, (1, 1, 128)), torch)
    api.kv_append_rope(q, kv, kv, kpd, vpd, to_dev(bt, torch), to_dev(lens, torch), 1e6, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) & 1
    assert np.array_equal(to_host(kpd), kp) and np.array_equal(to_host(vpd), vp)


# ----------------------------------------------------------------------------- attention

ATT_LENS = [1, 15, 16, 17, 31, 32, 33, 37, 200, 513]


@pytest.mark.parametrize("Hq,Hkv", [(7, 1), (28, 4), (8, 8), (16, 2)])
@pytest.mark.parametrize("part", [16, 64, 512, 0])
def test_paged_gqa_decode_matches_oracle(api, Hq, Hkv, part):
    r = np.random.default_rng(Hq * 100 + Hkv + part)
    D = 128
    lens = np.array(ATT_LENS, np.int32)
    B = len(lens)
    pages = int(sum((L + 15) // 16 for L in lens)) + 7
    kp = synth.kv_pool(r, pages, Hkv, D)
    vp = synth.kv_pool(r, pages, Hkv, D)
    bt = synth.block_table(r, lens, pages)
    q = synth.normal_fp16(r, (B, Hq, D), std=2.0)
    ref = orc.paged_attention(q, kp, vp, bt, lens, 1 / math.sqrt(D))
    out = api.paged_gqa_decode(to_dev(q, torch), to_dev(kp, torch), to_dev(vp, torch), to_dev(bt, torch),
                               to_dev(lens, torch), max_context=int(lens.max()), partition_tokens=part)
    torch.cuda.synchronize()
    assert_close(to_host(out), ref, what=f"attention Hq={Hq} Hkv={Hkv} part={part}")


def test_paged_gqa_decode_repeat_calls_and_zero_length(api):
    r = np.random.default_rng(11)
    D, Hq, Hkv = 128, 28, 4
    lens = np.array([0, 700, 64], np.int32)
    pages = 60
    kp = synth.kv_pool(r, pages, Hkv, D)
    vp = synth.kv_pool(r, pages, Hkv, D)
    bt = synth.block_table(r, lens, pages)
    q = synth.normal_fp16(r, (3, Hq, D))
    args = [to_dev(a, torch) for a in (q, kp, vp, bt, lens)]
    ws = torch.zeros(api.paged_gqa_decode_workspace_size(3, Hq, Hkv, 700, 64), dtype=torch.uint8, device="cuda")
    o1 = api.paged_gqa_decode(*args, max_context=700, partition_tokens=64, workspace=ws)
    o2 = api.paged_gqa_decode(*args, max_context=700, partition_tokens=64, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)  # the ticket counters were left at zero
    got = to_host(o1)
    assert np.all(got[0] == 0)
    ref = orc.paged_attention(q[1:], kp, vp, bt[1:], lens[1:], 1 / math.sqrt(D))
    assert_close(got[1:], ref, what="attention repeat")


def test_paged_gqa_decode_one_workspace_for_different_shapes(api):
    """Calls of different batch sizes and partition counts in turn on one
    workspace (the tickets sit at a fixed place whatever the shape)."""
    r = np.random.default_rng(13)
    D, Hq, Hkv = 128, 28, 4
    shapes = [(2, 5000, 16), (9, 1200, 16), (4, 3000, 32)]   # (B, max length, partition tokens)
    cases, need = [], 0
    for B, Lmax, part in shapes:
        lens = r.integers(1, Lmax + 1, size=B).astype(np.int32)
        lens[0] = Lmax
        pages = int(sum((L + 15) // 16 for L in lens)) + 3
        kp, vp = synth.kv_pool(r, pages, Hkv, D), synth.kv_pool(r, pages, Hkv, D)
        bt = synth.block_table(r, lens, pages)
        q = synth.normal_fp16(r, (B, Hq, D))
        ref = orc.paged_attention(q, kp, vp, bt, lens, 1 / math.sqrt(D))
        cases.append(([to_dev(a, torch) for a in (q, kp, vp, bt, lens)], Lmax, part, ref))
        need = max(need, api.paged_gqa_decode_workspace_size(B, Hq, Hkv, Lmax, part))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for rep in range(2):
        outs = [api.paged_gqa_decode(*args, max_context=Lmax, partition_tokens=part, workspace=ws)
                for args, Lmax, part, _ in cases]
        torch.cuda.synchronize()
        for o, (_, Lmax, part, ref) in zip(outs, cases):
            assert_close(to_host(o), ref, what=f"shared workspace pass {rep} part={part}")


def test_paged_gqa_decode_strided_q_matches_packed(api):
    r = np.random.default_rng(12)
    D, Hq, Hkv = 128, 28, 4
    lens = np.array([77, 300], np.int32)
    pages = 40
    kp = to_dev(synth.kv_pool(r, pages, Hkv, D), torch)
    vp = to_dev(synth.kv_pool(r, pages, Hkv, D), torch)
    bt = to_dev(synth.block_table(r, lens, pages), torch)
    ld = to_dev(lens, torch)
    row = to_dev(synth.normal_fp16(r, (2, (Hq + 2 * Hkv) * D)), torch)
    q_packed = row[:, :Hq * D].contiguous().view(2, Hq, D)
    a = api.paged_gqa_decode(q_packed, kp, vp, bt, ld, max_context=300, partition_tokens=64)
    b = api.paged_gqa_decode(row, kp, vp, bt, ld, max_context=300, partition_tokens=64, q_stride=row.shape[1],
                             n_q_heads=Hq)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_paged_gqa_decode_bad_page_flags_and_stays_finite(api):
    r = np.random.default_rng(13)
    D, Hq, Hkv = 128, 7, 1
    kp = synth.kv_pool(r, 8, Hkv, D)
    vp = synth.kv_pool(r, 8, Hkv, D)
    bt = np.array([[2, 123456, 5]], np.int32)
    lens = np.array([40], np.int32)
    q = synth.normal_fp16(r, (1, Hq, D))
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.paged_gqa_decode(to_dev(q, torch), to_dev(kp, torch), to_dev(vp, torch), to_dev(bt, torch),
                               to_dev(lens, torch), max_context=48, partition_tokens=16, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) & 1
    assert np.all(np.isfinite(to_host(out).astype(np.float64)))


# ----------------------------------------------------------------------------- embedding, lm_head

def test_embedding_gather_and_bad_token(api):
    r = np.random.default_rng(14)
    E = synth.normal_fp16(r, (300, 896))
    toks = np.array([0, 299, 17, 300], np.int32)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = api.embedding_gather(to_dev(E, torch), to_dev(toks, torch), err_flag=flag)
    torch.cuda.synchronize()
    got = to_host(x)
    for i in range(3):
        assert np.array_equal(got[i], E[toks[i]])
    assert np.all(got[3] == 0) and int(flag.item()) & 1


@pytest.mark.parametrize("B,H,V", [(1, 896, 5000), (3, 896, 4099), (1, 3584, 152064)])
def test_lm_head_argmax_matches_oracle(api, B, H, V):
    r = np.random.default_rng(B * H + V)
    W = synth.normal_fp16(r, (V, H), std=0.02)
    x = synth.normal_fp16(r, (B, H))
    toks, logits = api.lm_head_argmax(to_dev(x, torch), to_dev(W, torch), want_logits=True)
    torch.cuda.synchronize()
    toks, logits = to_host(toks), to_host(logits)
    for b in range(B):
        ref = orc.fp16_gemv(x[b], W)
        assert_close(logits[b], ref.astype(np.float16), what="lm_head logits")
        srt = np.sort(ref)
        if srt[-1] - srt[-2] > 4 * 1e-3:
            assert toks[b] == orc.argmax(ref)
        else:
            assert ref[toks[b]] >= srt[-1] - 4 * 1e-3


def test_lm_head_argmax_ties_take_lowest_index(api):
    H, V = 896, 3000
    W = np.zeros((V, H), np.float16)
    W[2999] = 1.0
    W[1234] = 1.0
    W[1235] = 1.0
    x = np.ones((1, H), np.float16)
    toks, _ = api.lm_head_argmax(to_dev(x, torch), to_dev(W, torch))
    torch.cuda.synchronize()
    assert int(to_host(toks)[0]) == 1234


@pytest.mark.parametrize("Hq,Hkv", [(7, 1), (28, 4)])
@pytest.mark.parametrize("part", [16, 64, 0])
def test_fused_rope_append_attention_matches_oracle(api, Hq, Hkv, part):
    r = np.random.default_rng(Hq * 7 + part)
    D, theta = 128, 1e6
    lens = np.array([1, 15, 16, 17, 31, 32, 33, 37, 513], np.int32)  # after the append
    B = len(lens)
    pages = int(sum((L + 15) // 16 for L in lens)) + 6
    kp = synth.kv_pool(r, pages, Hkv, D)
    vp = synth.kv_pool(r, pages, Hkv, D)
    bt = synth.block_table(r, lens, pages)
    qkv = synth.normal_fp16(r, (B, (Hq + 2 * Hkv) * D), std=2.0)
    q = qkv[:, :Hq * D].reshape(B, Hq, D)
    k = qkv[:, Hq * D:(Hq + Hkv) * D].reshape(B, Hkv, D)
    v = qkv[:, (Hq + Hkv) * D:].reshape(B, Hkv, D)
    q_rot = np.stack([orc.rope(q[b], int(lens[b]) - 1, theta) for b in range(B)])
    k_rot = np.stack([orc.rope(k[b], int(lens[b]) - 1, theta) for b in range(B)])
    kp_ref, vp_ref = kp.copy(), vp.copy()
    orc.kv_append(k_rot, v, kp_ref, vp_ref, bt, lens)
    ref = orc.paged_attention(q_rot, kp_ref, vp_ref, bt, lens, 1 / math.sqrt(D))
    kpd, vpd = to_dev(kp, torch), to_dev(vp, torch)
    qkvd = to_dev(qkv, torch)
    out = api.paged_gqa_decode_rope_append(qkvd, kpd, vpd, to_dev(bt, torch), to_dev(lens, torch),
                                           max_context=int(lens.max()), theta=theta, n_q_heads=Hq,
                                           partition_tokens=part)
    torch.cuda.synchronize()
    assert_close(to_host(out), ref, what=f"fused attention Hq={Hq} part={part}")
    kg, vg = to_host(kpd), to_host(vpd)
    assert np.array_equal(vg, vp_ref)                 # v placement and values bit-exact
    mask = np.zeros(kp.shape[:3], bool)
    for b in range(B):
        mask[bt[b, (lens[b] - 1) // 16], :, (lens[b] - 1) % 16] = True
    assert np.array_equal(kg[~mask], kp[~mask])        # nothing else moved
    assert_close(kg[mask], kp_ref[mask], what="appended k")
    assert np.array_equal(to_host(qkvd), qkv)         # q|k|v rows are read only


def test_paged_gqa_decode_batch32_mixed_lengths(api):
    """32 sequences with lengths U[1, 4096] (15/16/17 among them) and the
    library's partition choice (a warp per 256-token partition, partials
    combined by the last CTA of each sequence and kv head): every output
    against the oracle."""
    c = synth.QWEN_BATCHED
    r = synth.rng(4242)
    lens = synth.batched_lens(r, 32, 4096, c["forced_lens"]).astype(np.int32)
    Hq, Hkv, D = 28, 4, 128
    pages = int(sum((L + 15) // 16 for L in lens)) + 5
    kp = synth.kv_pool(r, pages, Hkv, D)
    vp = synth.kv_pool(r, pages, Hkv, D)
    bt = synth.block_table(r, lens, pages)
    q = synth.normal_fp16(r, (32, Hq, D), std=2.0)
    assert api.load().paged_gqa_decode_default_partition(32, Hkv, int(lens.max())) == 256
    out = api.paged_gqa_decode(to_dev(q, torch), to_dev(kp, torch), to_dev(vp, torch), to_dev(bt, torch),
                               to_dev(lens, torch), max_context=int(lens.max()))
    torch.cuda.synchronize()
    ref = orc.paged_attention(q, kp, vp, bt, lens, 1 / math.sqrt(D))
    assert_close(to_host(out), ref, what="attention b32 mixed lengths")
