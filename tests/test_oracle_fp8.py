"""Pins of the oracle's FP8 (E4M3) KV-page functions, on the CPU.

The E4M3 codec is checked against torch's float8_e4m3fn conversions (a
library implementation of the same format, independent of the oracle) on
all 256 codes and on random and tie values; saturation and the row
quantiser against closed forms; FP8 paged attention against the (already
pinned) fp16 paged attention on pools whose dequantised values are exactly
fp16."""
import numpy as np
import pytest

import oracle as orc
from w4a16_decode_paged_gb300 import synth

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    orc.build()


def _torch_decode(codes):
    t = torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def test_decode_all_256_codes_matches_library():
    codes = np.arange(256, dtype=np.uint8)
    ref = _torch_decode(codes)
    got = np.array([orc.e4m3_to_double(c) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got)) and nan.sum() == 2     # S.1111.111 only
    assert np.array_equal(got[~nan], ref[~nan])
    assert orc.e4m3_to_double(0x7E) == 448.0 and orc.e4m3_to_double(0x01) == 2.0 ** -9
    assert orc.e4m3_to_double(0x08) == 2.0 ** -6 and orc.e4m3_to_double(0x80) == 0.0


def test_encode_matches_library_on_random_values_and_ties():
    r = np.random.default_rng(5)
    vals = np.concatenate([
        r.standard_normal(20000).astype(np.float32) * np.float32(40.0),
        (r.random(5000).astype(np.float32) * np.float32(0.03)),           # subnormal range
        r.uniform(-448, 448, 5000).astype(np.float32),
    ])
    # midpoints between neighbouring codes: ties go to the even code
    finite = np.array([orc.e4m3_to_double(c) for c in range(0x7F) if c != 0x7F], np.float64)
    mids = ((finite[:-1] + finite[1:]) / 2).astype(np.float32)
    vals = np.concatenate([vals, mids, -mids]).astype(np.float32)
    vals = vals[np.abs(vals) <= 448]
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.float_to_e4m3(v) for v in vals], np.uint8)
    bad = np.flatnonzero(got != ref)
    # -0.0 vs +0.0 aside (torch keeps the sign of tiny negatives as well)
    assert bad.size == 0, [(float(vals[i]), int(got[i]), int(ref[i])) for i in bad[:5]]
    # every mid-point went to the code with an even fraction
    for m in mids[mids > 0]:
        assert orc.float_to_e4m3(float(m)) % 2 == 0


def test_encode_saturates_and_round_trips():
    assert orc.float_to_e4m3(448.0) == 0x7E
    assert orc.float_to_e4m3(463.9) == 0x7E and orc.float_to_e4m3(1e30) == 0x7E
    assert orc.float_to_e4m3(-500.0) == 0xFE
    for c in range(256):
        v = orc.e4m3_to_double(c)
        if np.isnan(v):
            continue
        assert orc.e4m3_to_double(orc.float_to_e4m3(v)) == v


def test_row_quantiser_maps_amax_to_448_within_half_a_step():
    r = np.random.default_rng(6)
    for scale_std in (1.0, 0.01, 30.0):
        x = synth.normal_fp16(r, (128,), std=scale_std)
        codes, sc = orc.fp8_quantize_row(x)
        xd = x.astype(np.float64)
        amax = np.max(np.abs(xd))
        assert sc == np.float32(np.float32(amax) / np.float32(448.0))
        deq = np.array([orc.e4m3_to_double(c) for c in codes]) * sc
        i = int(np.argmax(np.abs(xd)))
        assert abs(orc.e4m3_to_double(codes[i])) == 448.0
        # E4M3 normals have 3 fraction bits: relative rounding error <= 2^-4;
        # subnormal codes are spaced 2^-9 apart (absolute error <= 2^-10 * scale)
        err = np.abs(deq - xd)
        assert np.all(err <= np.maximum(np.abs(xd) * 2.0 ** -4, 2.0 ** -10 * sc) * (1 + 1e-6) + 1e-12)
    codes, sc = orc.fp8_quantize_row(np.zeros(128, np.float16))
    assert sc == 0.0 and np.all(codes == 0)


def test_append_fp8_touches_one_row_per_head():
    r = np.random.default_rng(7)
    pages, Hkv, D = 6, 2, 128
    kp = np.full((pages, Hkv, 16, D), 0x55, np.uint8)
    vp = kp.copy()
    ks = np.full((pages, Hkv, 16), -1.0, np.float32)
    vs = ks.copy()
    k = synth.normal_fp16(r, (1, Hkv, D))
    v = synth.normal_fp16(r, (1, Hkv, D))
    bt = np.array([[4, 1, 3]], np.int32)
    lens = np.array([18], np.int32)                    # position 17: page bt[1] = 1, slot 1
    kp0, ks0 = kp.copy(), ks.copy()
    orc.kv_append_fp8(k, v, kp, vp, ks, vs, bt, lens)
    changed = np.argwhere(np.any(kp != kp0, axis=-1))
    assert sorted(map(tuple, changed.tolist())) == [(1, 0, 1), (1, 1, 1)]
    assert np.array_equal(np.argwhere(ks != ks0), np.array([[1, 0, 1], [1, 1, 1]]))
    for h in range(Hkv):
        codes, sc = orc.fp8_quantize_row(k[0, h])
        assert np.array_equal(kp[1, h, 1], codes) and ks[1, h, 1] == np.float32(sc)


def test_fp8_paged_attention_equals_fp16_attention_on_exact_pools():
    """Pools whose rows have amax 448 * 2^-k (so the scale is a power of two)
    and values on the E4M3 grid: the dequantised rows are exactly fp16, and
    the FP8 attention must equal the fp16 attention on them bit for bit."""
    r = np.random.default_rng(8)
    pages, Hkv, Hq, D = 8, 2, 14, 128
    grid = np.array([orc.e4m3_to_double(c) for c in range(0x7F)], np.float64)   # non-negative finite codes
    codes = r.integers(0, 0x7F, size=(pages, Hkv, 16, D)).astype(np.uint8)
    sign = r.integers(0, 2, size=codes.shape).astype(np.uint8) << 7
    codes[..., 0] = 0x7E                                # each row's largest magnitude is 448
    kc = codes | sign
    vc = r.integers(0, 0x7F, size=codes.shape).astype(np.uint8)
    vc[..., 0] = 0x7E
    kexp = r.integers(-8, -2, size=(pages, Hkv, 16))
    vexp = r.integers(-8, -2, size=(pages, Hkv, 16))
    ks = (2.0 ** kexp).astype(np.float32)
    vs = (2.0 ** vexp).astype(np.float32)
    dec = lambda c: np.sign(0.5 - (c >> 7)) * grid[c & 0x7F]
    k16 = (dec(kc) * ks[..., None]).astype(np.float16)
    v16 = (dec(vc) * vs[..., None]).astype(np.float16)
    assert np.array_equal(k16.astype(np.float64), dec(kc) * ks[..., None])   # exactly representable
    lens = np.array([37, 5], np.int32)
    bt = synth.block_table(r, lens, pages)
    q = synth.normal_fp16(r, (2, Hq, D))
    got = orc.paged_attention_fp8(q, kc, vc, ks, vs, bt, lens, 1.0 / np.sqrt(D))
    ref = orc.paged_attention(q, k16, v16, bt, lens, 1.0 / np.sqrt(D))
    assert np.array_equal(got, ref)


def _fp8_pools(pool):
    """Quantise every row of an fp16 pool [pages][Hkv][16][D] with the
    (pinned) row quantiser: (codes uint8, scales fp32 [pages][Hkv][16])."""
    P, Hkv, T, D = pool.shape
    codes = np.zeros((P, Hkv, T, D), np.uint8)
    scales = np.zeros((P, Hkv, T), np.float32)
    for p in range(P):
        for h in range(Hkv):
            for t in range(T):
                codes[p, h, t], scales[p, h, t] = orc.fp8_quantize_row(pool[p, h, t])
    return codes, scales


def test_decoder_layer_over_fp8_pools_is_composition_of_pinned_parts():
    """A layer whose KV cache is FP8 pages: the same composition as the fp16
    layer with the FP8 append and the FP8 paged attention in place of the
    fp16 ones (each pinned above); only the appended rows of the pools
    change."""
    import math
    cfg = dict(synth.TINY_LAYER, bias=True)
    c = synth.layer_case(cfg, seed=1200)
    w = c["weights"]
    Hq, Hkv, D = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    L = int(c["context_lens"][0])
    k8, ks = _fp8_pools(c["k_pool"])
    v8, vs = _fp8_pools(c["v_pool"])
    k1, ks1, v1, vs1 = k8.copy(), ks.copy(), v8.copy(), vs.copy()
    out = orc.decoder_layer(cfg, w, c["x"], (k1, ks1), (v1, vs1), c["block_table"], c["context_lens"])

    k2, ks2, v2, vs2 = k8.copy(), ks.copy(), v8.copy(), vs.copy()
    xn = orc.rmsnorm(c["x"], w["ln1"], cfg["eps"])
    q = orc.rope(orc.w4a16_gemv(xn, w["wq"], w["sq"], bias=w["bq"]).reshape(Hq, D), L - 1, cfg["theta"])
    k = orc.rope(orc.w4a16_gemv(xn, w["wk"], w["sk"], bias=w["bk"]).reshape(Hkv, D), L - 1, cfg["theta"])
    v = orc.w4a16_gemv(xn, w["wv"], w["sv"], bias=w["bv"]).reshape(Hkv, D)
    orc.kv_append_fp8(k[None], v[None], k2, v2, ks2, vs2, c["block_table"], c["context_lens"])
    att = orc.paged_attention_fp8(q[None], k2, v2, ks2, vs2, c["block_table"], c["context_lens"], 1 / math.sqrt(D))
    h = orc.w4a16_gemv(att.reshape(1, Hq * D), w["wo"], w["so"], residual=c["x"])
    hn = orc.rmsnorm(h, w["ln2"], cfg["eps"])
    m = orc.silu_mul(orc.w4a16_gemv(hn, w["wg"], w["sg"]), orc.w4a16_gemv(hn, w["wu"], w["su"]))
    ref = orc.w4a16_gemv(m, w["wd"], w["sd"], residual=h)
    assert np.array_equal(out, ref)
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)
    assert np.array_equal(ks1, ks2) and np.array_equal(vs1, vs2)
    page, slot = int(c["block_table"][0, (L - 1) // 16]), (L - 1) % 16
    changed = {tuple(p) for p in np.argwhere(np.any(k1 != k8, axis=-1))}
    assert changed <= {(page, h, slot) for h in range(Hkv)}
    # the same layer over the fp16 pools differs (the cache really is FP8)
    out16 = orc.decoder_layer(cfg, w, c["x"], c["k_pool"].copy(), c["v_pool"].copy(), c["block_table"],
                              c["context_lens"])
    assert not np.array_equal(out, out16)
