"""Pins for the CPU oracle: each test ties an oracle function to something other
than itself (hand-derived fixtures, closed forms, invariants, library routines,
brute force on tiny inputs).  CPU only."""
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle as orc
from w4a16_decode_paged_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- fp16 codec

def test_half_to_double_all_bit_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    h = bits.view(np.float16)
    got = orc.half_to_double(h)
    ref = h.astype(np.float64)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_double_to_half_matches_numpy_rounding():
    r = np.random.default_rng(7)
    vals = np.concatenate([
        r.standard_normal(200000) * 10.0 ** r.integers(-9, 6, 200000),
        # exact ties between neighbouring halves, both parities
        (np.arange(0, 65536, dtype=np.uint32).astype(np.uint16).view(np.float16)[:0x7bff].astype(np.float64)
         + np.arange(1, 65536, dtype=np.uint32).astype(np.uint16).view(np.float16)[:0x7bff].astype(np.float64)) / 2,
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0**-24, 2.0**-25, 2.0**-25 * 1.0001,
                  6.1e-5, 2.0**-14, 2.0**-14 - 2.0**-25]),
    ])
    got = orc.double_to_half(vals).view(np.uint16)
    with np.errstate(over="ignore"):                 # values past 65520 round to inf on purpose
        ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- int4 format

def test_nibble_order_golden():
    for row in _read_golden("int4_nibble_order.txt"):
        word = int(row[0], 16)
        codes = [int(c) for c in row[1:]]
        assert [orc.unpack_code(word, i) for i in range(8)] == codes, row[0]
        packed = orc.pack_int4(np.array([codes], np.int8))
        assert int(packed[0, 0]) == word


def test_pack_unpack_roundtrip_all_codes_all_positions():
    # every code in every nibble position
    q = np.zeros((16 * 8, 8), np.int8) - 8
    for code in range(-8, 8):
        for pos in range(8):
            q[(code + 8) * 8 + pos, pos] = code
    assert np.array_equal(orc.unpack_int4(orc.pack_int4(q), 8), q)


def test_unpack_pack_roundtrip_random_words():
    r = np.random.default_rng(3)
    words = r.integers(0, 2**32, size=(1000, 1000), dtype=np.uint32)  # 10^6 words
    q = orc.unpack_int4(words, 8000)
    assert q.min() >= -8 and q.max() <= 7
    assert np.array_equal(orc.pack_int4(q), words)


def test_dequant_is_code_times_group_scale():
    r = np.random.default_rng(4)
    N, K = 6, 384
    q = r.integers(-8, 8, size=(N, K)).astype(np.int8)
    s = (2.0 ** r.integers(-8, 0, size=(N, K // 128))).astype(np.float16)
    w = orc.dequant(orc.pack_int4(q), s, K)
    # group g covers k in [128 g, 128 g + 128)
    for n in range(N):
        for g in range(K // 128):
            assert np.array_equal(w[n, 128 * g:128 * (g + 1)],
                                  q[n, 128 * g:128 * (g + 1)].astype(np.float64) * float(s[n, g]))


def test_quantize_recovers_exact_grid_weights():
    r = np.random.default_rng(5)
    N, K = 8, 256
    q = r.integers(-7, 8, size=(N, K)).astype(np.int8)
    q[:, 0] = 7  # makes amax/7 the exact scale of every group
    q[:, 128] = -7
    s = (2.0 ** r.integers(-9, -5, size=(N, K // 128))).astype(np.float16)
    w = q.astype(np.float64) * np.repeat(s.astype(np.float64), 128, axis=1)
    qw, s2 = orc.quantize(w)
    assert np.array_equal(s2, s)
    assert np.array_equal(orc.unpack_int4(qw, K), q)


# ---------------------------------------------------------------- GEMV

def test_gemv_one_hot_returns_codes():
    r = np.random.default_rng(6)
    N, K = 16, 256
    q = r.integers(-8, 8, size=(N, K)).astype(np.int8)
    qw = orc.pack_int4(q)
    s = np.ones((N, K // 128), np.float16)
    for k in (0, 1, 7, 8, 127, 128, 255):
        x = np.zeros((1, K), np.float16)
        x[0, k] = 1.0
        y = orc.w4a16_gemv(x, qw, s)
        assert np.array_equal(y[0].astype(np.float64), q[:, k].astype(np.float64))


def test_gemv_matches_numpy_matmul_on_dequantised_weights():
    r = np.random.default_rng(8)
    M, N, K = 3, 64, 896
    q = r.integers(-8, 8, size=(N, K)).astype(np.int8)
    s = r.uniform(0.005, 0.02, size=(N, K // 128)).astype(np.float16)
    x = r.standard_normal((M, K)).astype(np.float16)
    bias = (r.standard_normal(N) * 0.1).astype(np.float16)
    res = r.standard_normal((M, N)).astype(np.float16)
    wd = q.astype(np.float64) * np.repeat(s.astype(np.float64), 128, axis=1)   # built without the oracle
    ref = x.astype(np.float64) @ wd.T + bias.astype(np.float64) + res.astype(np.float64)
    y = orc.w4a16_gemv(x, orc.pack_int4(q), s, bias=bias, residual=res)
    diff = np.abs(y.astype(np.float64) - ref.astype(np.float16).astype(np.float64))
    ulp = np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64)
    assert np.all(diff <= ulp)  # at most one fp16 ulp (rounding of a different sum order)
    assert np.mean(diff == 0) > 0.99


def test_fp16_gemv_and_argmax():
    r = np.random.default_rng(9)
    w = r.standard_normal((50, 40)).astype(np.float16)
    x = r.standard_normal(40).astype(np.float16)
    out = orc.fp16_gemv(x, w)
    assert np.allclose(out, w.astype(np.float64) @ x.astype(np.float64), rtol=1e-12, atol=1e-12)
    v = np.array([1.0, 3.0, 3.0, -1.0, 3.0])
    assert orc.argmax(v) == 1  # lowest index on ties
    assert orc.argmax(np.array([-5.0])) == 0


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_constant_input_closed_form():
    H = 896
    for c in (0.5, 1.0, 3.0, -2.0):
        x = np.full((1, H), c, np.float16)
        g = np.linspace(0.5, 1.5, H).astype(np.float16)
        y = orc.rmsnorm(x, g, 1e-6)
        ref = (c / math.sqrt(c * c + 1e-6)) * g.astype(np.float64)
        assert np.array_equal(y[0], ref.astype(np.float16))


def test_rmsnorm_scale_invariance_and_unit_rms():
    r = np.random.default_rng(10)
    x = r.standard_normal((2, 3584)).astype(np.float16)
    g = np.ones(3584, np.float16)
    y1 = orc.rmsnorm(x, g, 0.0)
    y2 = orc.rmsnorm((x.astype(np.float32) * 4).astype(np.float16), g, 0.0)  # power of two: exact
    assert np.array_equal(y1, y2)
    rms = np.sqrt(np.mean(y1.astype(np.float64) ** 2, axis=1))
    assert np.allclose(rms, 1.0, atol=2e-3)


# ---------------------------------------------------------------- RoPE

def test_rope_inverse_frequency_closed_forms():
    assert orc.rope_inv_freq(0, 128, 1e6) == 1.0
    assert orc.rope_inv_freq(32, 128, 1e6) == np.float32(1e-3)   # 1e6^(-1/2)
    assert orc.rope_inv_freq(16, 128, 1e4) == np.float32(0.1)    # 1e4^(-1/4)
    assert orc.rope_angle(1, 5, 128, 1e6) == orc.rope_inv_freq(5, 128, 1e6)
    assert orc.rope_angle(0, 5, 128, 1e6) == 0.0
    # angle is the fp32 product, not the fp64 one
    a = orc.rope_angle(32767, 3, 128, 1e6)
    assert a == np.float32(np.float32(32767) * np.float32(orc.rope_inv_freq(3, 128, 1e6)))


def test_rope_position_zero_is_identity():
    r = np.random.default_rng(11)
    x = r.standard_normal((4, 128)).astype(np.float16)
    assert np.array_equal(orc.rope(x, 0, 1e6), x)


def test_rope_unit_vector_sign_and_pairing():
    D = 128
    for i in (0, 5, 63):
        x = np.zeros((1, D), np.float16)
        x[0, i] = 1.0                      # first half of pair i
        y = orc.rope(x, 7, 1e6).astype(np.float64)
        a = float(orc.rope_angle(7, i, D, 1e6))
        expect = np.zeros(D)
        expect[i], expect[i + D // 2] = math.cos(a), math.sin(a)
        assert np.allclose(y[0], expect.astype(np.float16).astype(np.float64), atol=0, rtol=0)


def test_rope_matches_complex_rotation_and_keeps_norm():
    r = np.random.default_rng(12)
    D, theta = 128, 1e6
    x = r.standard_normal((3, D)).astype(np.float16)
    for pos in (1, 17, 511, 32767):
        y = orc.rope(x, pos, theta).astype(np.float64)
        ang = np.array([orc.rope_angle(pos, i, D, theta) for i in range(D // 2)], np.float64)
        z = (x[:, :D // 2].astype(np.float64) + 1j * x[:, D // 2:].astype(np.float64)) * np.exp(1j * ang)
        ref = np.concatenate([z.real, z.imag], axis=1)
        assert np.allclose(y, ref.astype(np.float16).astype(np.float64), atol=2e-3, rtol=1e-3)
        n0 = np.hypot(x[:, :D // 2].astype(np.float64), x[:, D // 2:].astype(np.float64))
        n1 = np.hypot(y[:, :D // 2], y[:, D // 2:])
        assert np.allclose(n0, n1, atol=4e-3, rtol=2e-3)


def test_rope_composition_in_angle():
    # R(a) R(b) = R(a + b): rotating at pos p then at pos q equals pos p + q up to fp16 rounding
    r = np.random.default_rng(13)
    D, theta = 128, 1e6
    x = r.standard_normal((2, D)).astype(np.float16)
    y = orc.rope(orc.rope(x, 3, theta), 4, theta).astype(np.float64)
    z = orc.rope(x, 7, theta).astype(np.float64)
    assert np.allclose(y, z, atol=6e-3)


# ---------------------------------------------------------------- paging

def test_append_position_golden_and_single_slot():
    D, Hkv = 8, 2
    for row in _read_golden("paging_positions.txt"):
        L, pos, blk, slot = (int(v) for v in row)
        if L > 600:
            continue
        nblk = blk + 1
        pool_pages = nblk + 3
        bt = np.arange(pool_pages, dtype=np.int32)[::-1][:nblk].copy()[None, :]   # reversed ids
        kp = np.zeros((pool_pages, Hkv, 16, D), np.float16)
        vp = np.zeros_like(kp)
        k = np.ones((1, Hkv, D), np.float16)
        v = np.full((1, Hkv, D), 2.0, np.float16)
        orc.kv_append(k, v, kp, vp, bt, np.array([L], np.int32))
        nz = np.argwhere(kp != 0)
        assert len(nz) == Hkv * D
        assert set(nz[:, 0]) == {bt[0, blk]} and set(nz[:, 2]) == {slot}
        assert np.array_equal(np.argwhere(vp != 0), nz)


def test_paged_gather_with_shuffled_table_equals_contiguous():
    r = np.random.default_rng(14)
    Hkv, D, pages = 2, 16, 12
    for L in (1, 15, 16, 17, 31, 32, 33, 37):
        contig = r.standard_normal((pages * 16, Hkv, D)).astype(np.float16)   # token-major
        perm = r.permutation(pages).astype(np.int32)
        pool = np.zeros((pages, Hkv, 16, D), np.float16)
        for j in range(pages):
            pool[perm[j]] = contig[16 * j:16 * (j + 1)].transpose(1, 0, 2)
        got = orc.gather_kv(pool, perm, L)
        assert np.array_equal(got, contig[:L])


def _tiny_attention_case(r, Hq, Hkv, D, L):
    q = r.standard_normal((Hq, D)).astype(np.float16)
    k = r.standard_normal((L, Hkv, D)).astype(np.float16)
    v = r.standard_normal((L, Hkv, D)).astype(np.float16)
    return q, k, v


def test_attention_brute_force_tiny_vs_scipy_softmax():
    r = np.random.default_rng(15)
    for L in (1, 2, 3, 5):
        Hq, Hkv, D = 4, 2, 4
        q, k, v = _tiny_attention_case(r, Hq, Hkv, D, L)
        out = orc.attention(q, k, v, 0.5)
        for h in range(Hq):
            kh = h // 2
            s = np.array([sum(float(q[h, d]) * float(k[t, kh, d]) for d in range(D)) for t in range(L)]) * 0.5
            p = scipy.special.softmax(s)
            ref = sum(p[t] * v[t, kh].astype(np.float64) for t in range(L))
            assert np.array_equal(out[h], ref.astype(np.float16)) or np.allclose(out[h], ref, atol=1e-3)
            assert np.allclose(orc.attention_probs(q, k, 0.5, h), p, rtol=1e-12, atol=1e-15)


def test_attention_special_cases():
    r = np.random.default_rng(16)
    Hq, Hkv, D = 7, 1, 128
    # L = 1: output is v exactly
    q, k, v = _tiny_attention_case(r, Hq, Hkv, D, 1)
    out = orc.attention(q, k, v, 1 / math.sqrt(D))
    assert np.array_equal(out, np.repeat(v[0], Hq, axis=0))
    # all keys equal: output is the mean of v
    L = 37
    q, k, v = _tiny_attention_case(r, Hq, Hkv, D, L)
    k[:] = k[0]
    out = orc.attention(q, k, v, 1 / math.sqrt(D)).astype(np.float64)
    assert np.allclose(out, v.astype(np.float64).mean(axis=0)[0][None, :], atol=1e-3)
    # one dominant score selects its value row
    k = np.zeros((L, Hkv, D), np.float16)
    k[11, 0, :] = 1.0
    q = np.full((Hq, D), 1.0, np.float16)
    out = orc.attention(q, k, v, 1.0)
    assert np.array_equal(out, np.repeat(v[11], Hq, axis=0))
    # softmax rows sum to one
    q, k, v = _tiny_attention_case(r, Hq, Hkv, D, L)
    for h in range(Hq):
        assert abs(orc.attention_probs(q, k, 1 / math.sqrt(D), h).sum() - 1.0) < 1e-12


def test_paged_attention_shuffled_equals_contiguous():
    r = np.random.default_rng(17)
    Hq, Hkv, D, pages = 14, 2, 32, 40
    lens = np.array([1, 15, 16, 17, 31, 32, 33, 37], np.int32)
    pool_k = r.standard_normal((pages, Hkv, 16, D)).astype(np.float16)
    pool_v = r.standard_normal((pages, Hkv, 16, D)).astype(np.float16)
    bt = synth.block_table(r, lens, pages)
    q = r.standard_normal((len(lens), Hq, D)).astype(np.float16)
    out = orc.paged_attention(q, pool_k, pool_v, bt, lens, 0.2)
    for b, L in enumerate(lens):
        kc = np.concatenate([pool_k[bt[b, j]].transpose(1, 0, 2) for j in range((L + 15) // 16)])[:L]
        vc = np.concatenate([pool_v[bt[b, j]].transpose(1, 0, 2) for j in range((L + 15) // 16)])[:L]
        assert np.array_equal(out[b], orc.attention(q[b], kc, vc, 0.2))


def test_split_combine_equals_unsplit():
    r = np.random.default_rng(18)
    Hq, Hkv, D, L = 7, 1, 128, 1100
    q, k, v = _tiny_attention_case(r, Hq, Hkv, D, L)
    ref = orc.attention(q, k, v, 1 / math.sqrt(D)).astype(np.float64)
    for part in (16, 512, 2048):
        for h in (0, 3, 6):
            got = orc.attention_split_combine(q, k, v, 1 / math.sqrt(D), h, part)
            assert np.allclose(got, ref[h], atol=1e-3)


# ---------------------------------------------------------------- SiLU-mul

def test_silu_mul_matches_scipy_expit():
    r = np.random.default_rng(19)
    g = (r.standard_normal(10000) * 4).astype(np.float16)
    u = r.standard_normal(10000).astype(np.float16)
    ref = g.astype(np.float64) * scipy.special.expit(g.astype(np.float64)) * u.astype(np.float64)
    assert np.array_equal(orc.silu_mul(g, u), ref.astype(np.float16))
    assert orc.silu_mul(np.zeros(1, np.float16), np.ones(1, np.float16))[0] == 0


# ---------------------------------------------------------------- composition

def _tiny_layer_case(seed=1000):
    cfg = dict(synth.TINY_LAYER)
    return cfg, synth.layer_case(cfg, seed=seed)


def test_decoder_layer_is_composition_of_pinned_parts():
    cfg, c = _tiny_layer_case()
    w = c["weights"]
    H, Hq, Hkv, D = cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    L = int(c["context_lens"][0])
    kp1, vp1 = c["k_pool"].copy(), c["v_pool"].copy()
    out = orc.decoder_layer(cfg, w, c["x"], kp1, vp1, c["block_table"], c["context_lens"])

    kp2, vp2 = c["k_pool"].copy(), c["v_pool"].copy()
    xn = orc.rmsnorm(c["x"], w["ln1"], cfg["eps"])
    q = orc.w4a16_gemv(xn, w["wq"], w["sq"]).reshape(Hq, D)
    k = orc.w4a16_gemv(xn, w["wk"], w["sk"]).reshape(Hkv, D)
    v = orc.w4a16_gemv(xn, w["wv"], w["sv"]).reshape(Hkv, D)
    q = orc.rope(q, L - 1, cfg["theta"])
    k = orc.rope(k, L - 1, cfg["theta"])
    orc.kv_append(k[None], v[None], kp2, vp2, c["block_table"], c["context_lens"])
    att = orc.paged_attention(q[None], kp2, vp2, c["block_table"], c["context_lens"], 1 / math.sqrt(D))
    h = orc.w4a16_gemv(att.reshape(1, Hq * D), w["wo"], w["so"], residual=c["x"])
    hn = orc.rmsnorm(h, w["ln2"], cfg["eps"])
    m = orc.silu_mul(orc.w4a16_gemv(hn, w["wg"], w["sg"]), orc.w4a16_gemv(hn, w["wu"], w["su"]))
    ref = orc.w4a16_gemv(m, w["wd"], w["sd"], residual=h)
    assert np.array_equal(out, ref)
    assert np.array_equal(kp1, kp2) and np.array_equal(vp1, vp2)
    # only the appended slot changed in the pools
    changed = np.argwhere(np.any(kp1 != c["k_pool"], axis=-1))
    assert len(changed) <= Hkv and all(p[0] == c["block_table"][0, (L - 1) // 16] for p in changed)


def test_decode_step_zero_layers_is_norm_lm_head_argmax():
    r = np.random.default_rng(20)
    cfg = dict(synth.TINY_LAYER, vocab=300)
    H = cfg["hidden"]
    embed = r.standard_normal((cfg["vocab"], H)).astype(np.float16)
    lm = (r.standard_normal((cfg["vocab"], H)) * 0.02).astype(np.float16)
    fn = synth.gamma(r, H)
    toks = np.array([5, 299], np.int32)
    out, logits, hidden = orc.decode_step(cfg, [], [], [], embed, fn, lm, toks,
                                          np.zeros((2, 1), np.int32), np.ones(2, np.int32),
                                          n_layers_run=0, want_logits=True)
    for b, t in enumerate(toks):
        assert np.array_equal(hidden[b], embed[t])
        ref = orc.fp16_gemv(orc.rmsnorm(embed[t], fn, cfg["eps"])[0], lm)
        assert out[b] == int(np.argmax(ref))
        assert np.array_equal(logits[b], ref.astype(np.float16))


def test_decoder_layer_with_bias_and_two_sequences():
    """The composition pin again with the q/k/v biases on and two sequences
    whose new tokens land at a page's last slot (L = 16) and first slot
    (L = 17), each sequence composed on its own."""
    cfg = dict(synth.TINY_LAYER, bias=True, batch=2, pool_pages=8)
    c = synth.layer_case(cfg, lens=[16, 17], seed=1010)
    w = c["weights"]
    assert w["bq"] is not None and np.any(w["bq"] != 0)
    Hq, Hkv, D = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    kp1, vp1 = c["k_pool"].copy(), c["v_pool"].copy()
    out = orc.decoder_layer(cfg, w, c["x"], kp1, vp1, c["block_table"], c["context_lens"])
    kp2, vp2 = c["k_pool"].copy(), c["v_pool"].copy()
    for b in range(2):
        L = int(c["context_lens"][b])
        bt, lens = c["block_table"][b:b + 1], c["context_lens"][b:b + 1]
        xn = orc.rmsnorm(c["x"][b:b + 1], w["ln1"], cfg["eps"])
        q = orc.rope(orc.w4a16_gemv(xn, w["wq"], w["sq"], bias=w["bq"]).reshape(Hq, D), L - 1, cfg["theta"])
        k = orc.rope(orc.w4a16_gemv(xn, w["wk"], w["sk"], bias=w["bk"]).reshape(Hkv, D), L - 1, cfg["theta"])
        v = orc.w4a16_gemv(xn, w["wv"], w["sv"], bias=w["bv"]).reshape(Hkv, D)
        orc.kv_append(k[None], v[None], kp2, vp2, bt, lens)
        att = orc.paged_attention(q[None], kp2, vp2, bt, lens, 1 / math.sqrt(D))
        h = orc.w4a16_gemv(att.reshape(1, Hq * D), w["wo"], w["so"], residual=c["x"][b:b + 1])
        hn = orc.rmsnorm(h, w["ln2"], cfg["eps"])
        m = orc.silu_mul(orc.w4a16_gemv(hn, w["wg"], w["sg"]), orc.w4a16_gemv(hn, w["wu"], w["su"]))
        ref = orc.w4a16_gemv(m, w["wd"], w["sd"], residual=h)
        assert np.array_equal(out[b], ref[0]), f"sequence {b}"
    assert np.array_equal(kp1, kp2) and np.array_equal(vp1, vp2)
    # the biases matter: without them the layer output differs
    w0 = dict(w, bq=None, bk=None, bv=None)
    out0 = orc.decoder_layer(cfg, w0, c["x"], c["k_pool"].copy(), c["v_pool"].copy(), c["block_table"],
                             c["context_lens"])
    assert not np.array_equal(out0, out)


def test_decode_step_one_layer_is_embedding_layer_norm_lm_head_argmax():
    cfg = dict(synth.TINY_LAYER, vocab=97, n_layers=1)
    case = synth.model_case(cfg, lens=[20, 31], gen_tokens=2, pool_pages=8, seed=1020)
    lens = case["lens"] + 1                                  # counts after this step's append
    kp, vp = synth.host_pool(case, 0, "k"), synth.host_pool(case, 0, "v")
    toks, logits, hidden = orc.decode_step(cfg, case["layers"], [kp.copy()], [vp.copy()], case["embed"],
                                           case["fnorm"], case["lm"], case["tok"], case["bt"], lens,
                                           want_logits=True)
    x = orc.decoder_layer(cfg, case["layers"][0], case["embed"][case["tok"]], kp, vp, case["bt"], lens)
    assert np.array_equal(hidden, x)
    for b in range(2):
        ref = orc.fp16_gemv(orc.rmsnorm(x[b], case["fnorm"], cfg["eps"])[0], case["lm"])
        assert np.array_equal(logits[b], ref.astype(np.float16))
        assert toks[b] == orc.argmax(ref)
