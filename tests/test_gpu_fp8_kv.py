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


def _fp8_of_pool(pool):
    """The oracle's row quantiser over a whole fp16 pool [pages][Hkv][16][D]."""
    codes = np.zeros(pool.shape, np.uint8)
    scales = np.zeros(pool.shape[:3], np.float32)
    for idx in np.ndindex(pool.shape[:3]):
        if np.any(pool[idx] != 0):
            codes[idx], scales[idx] = orc.fp8_quantize_row(pool[idx])
    return codes, scales


def _fp8_model(api, case, max_context):
    cfg = case["cfg"]
    host, dls = [], []
    for l, w in enumerate(case["layers"]):
        k8, ks = _fp8_of_pool(synth.host_pool(case, l, "k"))
        v8, vs = _fp8_of_pool(synth.host_pool(case, l, "v"))
        host.append(((k8, ks), (v8, vs)))
        dls.append(api.device_layer(w, (k8, ks), (v8, vs)))
    m = api.Model(cfg, dls, embed=to_dev(case["embed"], torch), final_norm=to_dev(case["fnorm"], torch),
                  lm_head=to_dev(case["lm"], torch), max_batch=case["tok"].size, max_context=max_context,
                  num_pages=case["pool_pages"])
    return m, dls, host


def test_fp8_model_decode_free_running_matches_oracle(api):
    """A 3-layer model whose KV cache is FP8 pages: 10 free-running greedy
    steps of decode_step against the oracle's decode over FP8 pools (the same
    codes and scales to start with; each side appends its own quantised rows)."""
    cfg = dict(synth.TINY_LAYER, n_layers=3, vocab=900, bias=True, codes="symmetric")
    case = synth.model_case(cfg, lens=[37], gen_tokens=16, pool_pages=32, seed=9900)
    m, dls, host = _fp8_model(api, case, 128)
    assert m.decode_path(1) == "kernels"   # the persistent kernel is not built for FP8 pools
    tok = to_dev(case["tok"], torch)
    ld = to_dev(case["lens"], torch)
    btd = to_dev(case["bt"], torch)
    logits = torch.empty((1, cfg["vocab"]), dtype=torch.float16, device="cuda")
    kps = [h[0] for h in host]
    vps = [h[1] for h in host]
    t_or, n = case["tok"].copy(), case["lens"].copy()
    for step in range(10):
        fed = to_host(tok).astype(np.int32).copy()
        m.decode_step(tok, tok, btd, ld, logits=logits, use_graph=True)
        n = n + 1
        t_next, lg, _ = orc.decode_step(cfg, case["layers"], kps, vps, case["embed"], case["fnorm"], case["lm"],
                                        fed, case["bt"], n, want_logits=True)
        got, ref = to_host(logits)[0].astype(np.float64), lg[0].astype(np.float64)
        rel = np.sqrt(np.mean((got - ref) ** 2) / np.mean(ref ** 2))
        assert rel < 0.03, f"step {step}: logits differ by {rel:.3g} of their RMS"
        srt = np.sort(ref)
        if srt[-1] - srt[-2] > 4 * float(np.max(np.abs(got - ref))) + 2e-3:
            assert int(to_host(tok)[0]) == int(t_next[0]), f"step {step}"
    assert m.check_errors() == 0
    # the appended rows are FP8: every new position's scale is set, codes decode near the oracle's rows
    pos = np.arange(int(case["lens"][0]), int(n[0]))
    pages, slots = case["bt"][0, pos // 16], pos % 16
    for l in range(cfg["n_layers"]):
        vs_dev = to_host(dls[l]["v_scale"])[pages, :, slots]
        assert np.all(vs_dev > 0)
        v_dev = np.vectorize(orc.e4m3_to_double)(to_host(dls[l]["v8"])[pages, :, slots]) * vs_dev[..., None]
        v_ref = np.vectorize(orc.e4m3_to_double)(vps[l][0][pages, :, slots]) * vps[l][1][pages, :, slots][..., None]
        rel = np.sqrt(np.mean((v_dev - v_ref) ** 2) / np.mean(v_ref ** 2))
        assert rel < 0.05, f"layer {l}: appended v rows differ by {rel:.3g} of their RMS"
    m.close()


def test_fp8_model_batched_step(api):
    """Four sequences on FP8 pools (the CUDA-core batch path) for two steps
    against the oracle."""
    cfg = dict(synth.TINY_LAYER, n_layers=2, vocab=700, bias=True, codes="symmetric")
    case = synth.model_case(cfg, lens=[1, 16, 17, 40], gen_tokens=4, pool_pages=32, seed=9910)
    m, dls, host = _fp8_model(api, case, 64)
    tok = to_dev(case["tok"], torch)
    ld = to_dev(case["lens"], torch)
    logits = torch.empty((4, cfg["vocab"]), dtype=torch.float16, device="cuda")
    kps = [h[0] for h in host]
    vps = [h[1] for h in host]
    n = case["lens"].copy()
    for step in range(2):
        fed = to_host(tok).astype(np.int32).copy()
        m.decode_step(tok, tok, to_dev(case["bt"], torch), ld, logits=logits, use_graph=False)
        n = n + 1
        _, lg, _ = orc.decode_step(cfg, case["layers"], kps, vps, case["embed"], case["fnorm"], case["lm"],
                                   fed, case["bt"], n, want_logits=True)
        got, ref = to_host(logits).astype(np.float64), lg.astype(np.float64)
        rel = np.sqrt(np.mean((got - ref) ** 2) / np.mean(ref ** 2))
        assert rel < 0.03, f"step {step}: logits differ by {rel:.3g} of their RMS"
    assert m.check_errors() == 0
    m.close()


@pytest.mark.parametrize("cached,T", [(0, 37), (21, 16)])
def test_fp8_prefill_matches_oracle_token_by_token(api, cached, T):
    """w4a16_prefill over FP8 pools (quantised append of every prompt row,
    the causal prompt attention over the codes) against the oracle feeding
    the prompt one token per decode step over the same FP8 pools: last-token
    logits, and the appended rows (scales set, values close)."""
    cfg = dict(synth.TINY_LAYER, n_layers=2, vocab=800, bias=True, codes="symmetric")
    case = synth.model_case(cfg, lens=[cached], gen_tokens=T + 2, pool_pages=(cached + T) // 16 + 8,
                            seed=9920 + cached)
    prompt = synth.rng(9921 + cached).integers(0, cfg["vocab"], size=T).astype(np.int32)
    m, dls, host = _fp8_model(api, case, cached + T + 16)
    ld = to_dev(case["lens"], torch)
    logits = torch.empty((1, cfg["vocab"]), dtype=torch.float16, device="cuda")
    tok = m.prefill(to_dev(prompt, torch), to_dev(case["bt"], torch), ld, logits=logits)
    torch.cuda.synchronize()
    assert m.check_errors() == 0
    assert int(to_host(ld)[0]) == cached + T
    kps = [h[0] for h in host]
    vps = [h[1] for h in host]
    for i, tk in enumerate(prompt):
        t_next, lg, _ = orc.decode_step(cfg, case["layers"], kps, vps, case["embed"], case["fnorm"], case["lm"],
                                        np.array([tk], np.int32), case["bt"], np.array([cached + i + 1], np.int32),
                                        want_logits=True)
    got, ref = to_host(logits)[0].astype(np.float64), lg[0].astype(np.float64)
    rel = np.sqrt(np.mean((got - ref) ** 2) / np.mean(ref ** 2))
    assert rel < 0.03, f"logits differ by {rel:.3g} of their RMS"
    srt = np.sort(ref)
    if srt[-1] - srt[-2] > 4 * float(np.max(np.abs(got - ref))) + 2e-3:
        assert int(to_host(tok)[0]) == int(t_next[0])
    pos = np.arange(cached, cached + T)
    pages, slots = case["bt"][0, pos // 16], pos % 16
    dec = np.vectorize(orc.e4m3_to_double)
    for l in range(cfg["n_layers"]):
        for name, (codes, scales) in (("k", kps[l]), ("v", vps[l])):
            sd = to_host(dls[l][name + "_scale"])[pages, :, slots]
            assert np.all(sd > 0), (l, name)
            got_rows = dec(to_host(dls[l][name + "8"])[pages, :, slots]) * sd[..., None]
            ref_rows = dec(codes[pages, :, slots]) * scales[pages, :, slots][..., None]
            rel = np.sqrt(np.mean((got_rows - ref_rows) ** 2) / np.mean(ref_rows ** 2))
            assert rel < 0.05, f"layer {l} {name}: prompt rows differ by {rel:.3g} of their RMS"
    m.close()
