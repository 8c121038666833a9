"""w4a16_prefill (a prompt in one pass) against the CPU oracle fed the same
prompt one token at a time through its decode step: the next token and the
last token's logits, and the KV rows written for every prompt position
(placement exact; values to the composite bound).  Then decoding continues
from the prefilled cache.  GPU only (marked gpu)."""
import numpy as np
import pytest

import oracle as orc
from gpu_util import to_dev, to_host
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


def _rms_rel(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    return float(np.sqrt(np.mean((got - ref) ** 2) / np.mean(ref ** 2)))


def _case(cfg, cached, T, extra, seed):
    case = synth.model_case(cfg, lens=[cached], gen_tokens=T + extra, pool_pages=(cached + T + extra) // 16 + 8,
                            seed=seed)
    r = synth.rng(seed + 1)
    prompt = r.integers(0, cfg["vocab"], size=T).astype(np.int32)
    return case, prompt


def _prefill_vs_oracle(api, cfg, cached, T, seed, decode_after=0, rel_bound=0.02):
    case, prompt = _case(cfg, cached, T, decode_after + 1, seed)
    L = cfg["n_layers"]
    dls = [api.device_layer(w, api.device_pool(case, l, "k"), api.device_pool(case, l, "v"))
           for l, w in enumerate(case["layers"])]
    m = api.Model(cfg, dls, embed=to_dev(case["embed"], torch), final_norm=to_dev(case["fnorm"], torch),
                  lm_head=to_dev(case["lm"], torch), max_batch=1, max_context=cached + T + decode_after + 16,
                  num_pages=case["pool_pages"])
    btd = to_dev(case["bt"], torch)
    ld = to_dev(case["lens"], torch)
    logits = torch.empty((1, cfg["vocab"]), dtype=torch.float16, device="cuda")
    tok = m.prefill(to_dev(prompt, torch), btd, ld, logits=logits)
    torch.cuda.synchronize()
    assert m.check_errors() == 0
    assert int(to_host(ld)[0]) == cached + T
    # the oracle: the prompt one token per decode step
    kps = [synth.host_pool(case, l, "k") for l in range(L)]
    vps = [synth.host_pool(case, l, "v") for l in range(L)]
    k0 = [k.copy() for k in kps]
    for i, t in enumerate(prompt):
        t_next, lg, _ = orc.decode_step(cfg, case["layers"], kps, vps, case["embed"], case["fnorm"], case["lm"],
                                        np.array([t], np.int32), case["bt"], np.array([cached + i + 1], np.int32),
                                        want_logits=True)
    got_lg = to_host(logits)[0].astype(np.float64)
    ref_lg = lg[0].astype(np.float64)
    assert _rms_rel(got_lg, ref_lg) < rel_bound, f"logits differ by {_rms_rel(got_lg, ref_lg):.3g} of their RMS"
    srt = np.sort(ref_lg)
    if srt[-1] - srt[-2] > 4 * float(np.max(np.abs(got_lg - ref_lg))) + 2e-3:
        assert int(to_host(tok)[0]) == int(t_next[0])
    # KV rows: exactly the prompt positions changed; values close to the oracle's
    pos = np.arange(cached, cached + T)
    pages, slots = case["bt"][0, pos // 16], pos % 16
    for l in range(L):
        for name, ref_pool in (("k_pool", kps[l]), ("v_pool", vps[l])):
            got = to_host(dls[l][name])
            diff = np.any(got != k0[l] if name == "k_pool" else got != synth.host_pool(case, l, "v"), axis=-1)
            moved = {(int(p), int(s)) for p, _, s in np.argwhere(diff)}
            assert moved <= set(zip(pages.tolist(), slots.tolist())), (l, name)
            rel = _rms_rel(got[pages, :, slots], ref_pool[pages, :, slots])
            assert rel < rel_bound, f"layer {l} {name}: rows differ by {rel:.3g} of their RMS"
    # decoding continues from the prefilled cache; the oracle is fed the
    # device's tokens (near-ties may pick either), logits compared each step
    if decode_after:
        n = np.array([cached + T], np.int32)
        for step in range(decode_after):
            fed = to_host(tok).astype(np.int32).copy()
            m.decode_step(tok, tok, btd, ld, logits=logits, use_graph=True)
            n = n + 1
            t_nx, lg, _ = orc.decode_step(cfg, case["layers"], kps, vps, case["embed"], case["fnorm"], case["lm"],
                                          fed, case["bt"], n, want_logits=True)
            g, r = to_host(logits)[0].astype(np.float64), lg[0].astype(np.float64)
            assert _rms_rel(g, r) < rel_bound, f"decode step {step} after prefill"
            srt = np.sort(r)
            if srt[-1] - srt[-2] > 4 * float(np.max(np.abs(g - r))) + 2e-3:
                assert int(to_host(tok)[0]) == int(t_nx[0])
        assert m.check_errors() == 0
    m.close()


@pytest.mark.parametrize("cached,T", [(0, 1), (0, 16), (0, 37), (5, 40), (31, 33)])
def test_prefill_tiny_matches_oracle(api, cached, T):
    cfg = dict(synth.TINY_LAYER, n_layers=2, vocab=800, bias=True, codes="symmetric")
    _prefill_vs_oracle(api, cfg, cached, T, seed=9500 + 7 * cached + T)


def test_prefill_then_decode_continues(api):
    cfg = dict(synth.TINY_LAYER, n_layers=2, vocab=800, bias=True, codes="symmetric")
    _prefill_vs_oracle(api, cfg, 0, 45, seed=9600, decode_after=6)


def test_prefill_qwen_width_one_layer(api):
    """Qwen2.5-7B widths, one layer, a 64-token prompt (several row chunks
    of the tensor-core GEMMs and page boundaries)."""
    cfg = dict(synth.QWEN_MODEL, n_layers=1)
    _prefill_vs_oracle(api, cfg, 0, 64, seed=9700, rel_bound=0.01)
