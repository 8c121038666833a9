"""FP8 (E4M3) KV pages on the GPU against the CPU oracle: the quantised
append (codes bit-exact where no rounding of the rotation intervenes, else
within one code step), paged attention over FP8 pools (fp16 bound), and the
fused RoPE + append + attention.  GPU only (marked gpu)."""
import math

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
    orc.build()
    return _api


def _fp8_pools(r, pages, Hkv, D=128):
    """Random FP8 pools: every row quantised by the oracle from N(0,1) fp16
    rows with a per-row spread, so codes and scales are what appends make."""
    k = synth.normal_fp16(r, (pages, Hkv, 16, D)) * np.float16(2.0)
    v = synth.normal_fp16(r, (pages, Hkv, 16, D))
    kc = np.empty(k.shape, np.uint8)
    vc = np.empty(v.shape, np.uint8)
    ks = np.empty(k.shape[:3], np.float32)
    vs = np.empty(v.shape[:3], np.float32)
    for idx in np.ndindex(k.shape[:3]):
        kc[idx], ks[idx] = orc.fp8_quantize_row(k[idx])
        vc[idx], vs[idx] = orc.fp8_quantize_row(v[idx])
    return kc, vc, ks, vs


def _dev(torch_, *arrs):
    return [to_dev(a, torch_) for a in arrs]


@pytest.mark.parametrize("G,lens,part", [(7, [1, 15, 16, 17, 37, 513], 0), (7, [2000, 33], 64),
                                         (4, [300, 1000, 1], 128), (1, [77], 16)])
def test_fp8_paged_attention_matches_oracle(api, G, lens, part):
    r = np.random.default_rng(9000 + G + len(lens))
    Hkv = 4 if G != 1 else 2
    Hq, D = G * Hkv, 128
    lens = np.asarray(lens, np.int32)
    pages = int(sum((L + 15) // 16 for L in lens)) + 5
    kc, vc, ks, vs = _fp8_pools(r, pages, Hkv)
    bt = synth.block_table(r, lens, pages)
    q = synth.normal_fp16(r, (len(lens), Hq, D))
    max_ctx = int(lens.max())
    out = api.paged_gqa_decode_fp8(*_dev(torch, q, kc, vc, ks, vs, bt, lens), max_context=max_ctx,
                                   partition_tokens=part)
    ref = orc.paged_attention_fp8(q, kc, vc, ks, vs, bt, lens, 1.0 / math.sqrt(D))
    assert_close(to_host(out), ref, what=f"fp8 attention G={G}")


def test_fp8_long_context_attention_b4_ctx32768(api):
    """The long-context workload (4 x 32768 tokens, 512-token partitions)
    with FP8 pages: all outputs."""
    c = synth.QWEN_LONG
    r = np.random.default_rng(9100)
    B, Hq, Hkv, D, L, pool = c["batch"], c["n_q_heads"], c["n_kv_heads"], c["head_dim"], c["context"], 8200
    # pools quantised on the device side of the test by the oracle's rule is too slow at
    # this size; draw codes and scales directly (any codes are valid pages)
    kc = r.integers(0, 256, size=(pool, Hkv, 16, D), dtype=np.uint8)
    vc = r.integers(0, 256, size=(pool, Hkv, 16, D), dtype=np.uint8)
    for a in (kc, vc):
        a[(a & 0x7F) == 0x7F] = 0x7E                 # no NaN codes
    ks = r.uniform(0.001, 0.01, size=(pool, Hkv, 16)).astype(np.float32)
    vs = r.uniform(0.001, 0.01, size=(pool, Hkv, 16)).astype(np.float32)
    lens = np.full(B, L, np.int32)
    bt = synth.block_table(r, lens, pool)
    q = synth.normal_fp16(r, (B, Hq, D))
    out = api.paged_gqa_decode_fp8(*_dev(torch, q, kc, vc, ks, vs, bt, lens), max_context=L,
                                   partition_tokens=c["partition_tokens"])
    ref = orc.paged_attention_fp8(q, kc, vc, ks, vs, bt, lens, 1.0 / math.sqrt(D))
    assert_close(to_host(out), ref, what="fp8 b4 ctx32768")


@pytest.mark.parametrize("lens", [[1], [16, 17], [37, 512, 2]])
def test_fp8_append_rope(api, lens):
    r = np.random.default_rng(9200 + sum(lens))
    Hq, Hkv, D, theta = 14, 2, 128, 1e6
    lens = np.asarray(lens, np.int32)
    B = len(lens)
    pages = int(sum((L + 15) // 16 for L in lens)) + 3
    kc = np.full((pages, Hkv, 16, D), 0x33, np.uint8)
    vc = kc.copy()
    ks = np.full((pages, Hkv, 16), -1.0, np.float32)
    vs = ks.copy()
    bt = synth.block_table(r, lens, pages)
    q = synth.normal_fp16(r, (B, Hq, D))
    k = synth.normal_fp16(r, (B, Hkv, D))
    v = synth.normal_fp16(r, (B, Hkv, D))
    dq, dk, dv, dkc, dvc, dks, dvs, dbt, dl = _dev(torch, q, k, v, kc, vc, ks, vs, bt, lens)
    api.kv_append_rope_fp8(dq, dk, dv, dkc, dvc, dks, dvs, dbt, dl, theta)
    torch.cuda.synchronize()
    gkc, gvc, gks, gvs = to_host(dkc), to_host(dvc), to_host(dks), to_host(dvs)
    # placement: exactly one row per (sequence, kv head) changed
    rows = {(int(bt[b, (L - 1) // 16]), (L - 1) % 16) for b, L in enumerate(lens)}
    for name, got, before in (("k", gkc, kc), ("v", gvc, vc)):
        changed = np.argwhere(np.any(got != before, axis=-1))
        assert {(int(p), int(s)) for p, _, s in changed} <= rows, name
    # v: no rotation, so the codes and scales are the oracle's exactly
    ref_kc, ref_vc, ref_ks, ref_vs = kc.copy(), vc.copy(), ks.copy(), vs.copy()
    k_rot = np.stack([orc.rope(k[b], int(L) - 1, theta) for b, L in enumerate(lens)])
    orc.kv_append_fp8(k_rot, v, ref_kc, ref_vc, ref_ks, ref_vs, bt, lens)
    assert np.array_equal(gvc, ref_vc) and np.array_equal(gvs, ref_vs)
    # k: rotated in fp32 on the device, fp64 in the oracle, each rounded to
    # fp16 before quantising; equal where the fp16 rotations agree, and the
    # dequantised rows always within one code step
    deq = lambda c, s: np.vectorize(orc.e4m3_to_double)(c) * s[..., None]
    for b, L in enumerate(lens):
        p, sl = int(bt[b, (L - 1) // 16]), (L - 1) % 16
        got = deq(gkc[p, :, sl], gks[p, :, sl])
        ref = deq(ref_kc[p, :, sl], ref_ks[p, :, sl])
        assert np.all(np.abs(got - ref) <= 2.0 ** -3 * np.abs(ref) + 2.0 ** -9 * ref_ks[p, :, sl, None] * 1.01)
        if L == 1:  # position 0: the rotation is the identity, nothing rounds
            assert np.array_equal(gkc[p, :, sl], ref_kc[p, :, sl])
    # q rotated in place
    assert_close(to_host(dq), np.stack([orc.rope(q[b], int(L) - 1, theta) for b, L in enumerate(lens)]), what="q")


@pytest.mark.parametrize("lens,part", [([37], 0), ([16, 513, 1], 64), ([1000, 3000], 512)])
def test_fp8_fused_rope_append_attention(api, lens, part):
    r = np.random.default_rng(9300 + sum(lens))
    Hq, Hkv, D, theta = 28, 4, 128, 1e6
    lens = np.asarray(lens, np.int32)
    B = len(lens)
    pages = int(sum((L + 15) // 16 for L in lens)) + 4
    kc, vc, ks, vs = _fp8_pools(r, pages, Hkv)
    bt = synth.block_table(r, lens, pages)
    qkv = synth.normal_fp16(r, (B, (Hq + 2 * Hkv) * D))
    dqkv, dkc, dvc, dks, dvs, dbt, dl = _dev(torch, qkv, kc, vc, ks, vs, bt, lens)
    out = api.paged_gqa_decode_fp8(dqkv, dkc, dvc, dks, dvs, dbt, dl, max_context=int(lens.max()),
                                   partition_tokens=part, qkv_theta=theta, n_q_heads=Hq)
    torch.cuda.synchronize()
    gkc, gvc, gks, gvs = to_host(dkc), to_host(dvc), to_host(dks), to_host(dvs)
    # the attention the oracle computes on the device's own pools (after its
    # append) with the oracle's rotation of q
    q = qkv[:, :Hq * D].reshape(B, Hq, D)
    q_rot = np.stack([orc.rope(q[b], int(L) - 1, theta) for b, L in enumerate(lens)])
    ref = orc.paged_attention_fp8(q_rot, gkc, gvc, gks, gvs, bt, lens, 1.0 / math.sqrt(D))
    assert_close(to_host(out), ref, what="fused fp8 attention")
    # the appended v rows are the oracle's quantisation exactly; nothing else moved
    v_new = qkv[:, (Hq + Hkv) * D:].reshape(B, Hkv, D)
    for b, L in enumerate(lens):
        p, sl = int(bt[b, (L - 1) // 16]), (L - 1) % 16
        for h in range(Hkv):
            codes, sc = orc.fp8_quantize_row(v_new[b, h])
            assert np.array_equal(gvc[p, h, sl], codes) and gvs[p, h, sl] == np.float32(sc)
    rows = {(int(bt[b, (L - 1) // 16]), (L - 1) % 16) for b, L in enumerate(lens)}
    changed = np.argwhere(np.any(gkc != kc, axis=-1))
    assert {(int(p), int(s)) for p, _, s in changed} <= rows
