"""The persistent decode kernel (one cooperative launch per token) against
the CPU oracle and against the kernel-per-operation path.  GPU only (marked
gpu).

With one decoder layer the layer's input is the embedding row, so every
phase of the persistent step is checked elementwise on its own device
inputs (the activations it leaves in the model's arena), exactly as the
per-kernel tests check model.layer."""
import numpy as np
import pytest

import oracle as orc
from gpu_util import assert_close, check_layer_kernels, to_dev, to_host
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


def _model(api, case, max_context, path="persistent"):
    cfg = case["cfg"]
    dls = [api.device_layer(w, api.device_pool(case, l, "k"), api.device_pool(case, l, "v"))
           for l, w in enumerate(case["layers"])]
    m = api.Model(cfg, dls, embed=to_dev(case["embed"], torch), final_norm=to_dev(case["fnorm"], torch),
                  lm_head=to_dev(case["lm"], torch), max_batch=1, max_context=max_context,
                  num_pages=case["pool_pages"])
    m.set_decode_path(path)
    return m, dls


def _one_layer_every_phase(api, case, max_context):
    cfg = case["cfg"]
    m, dls = _model(api, case, max_context)
    assert m.decode_path(1) == "persistent" and m.kernel_count(1) == 1
    tok = to_dev(case["tok"], torch)
    ld = to_dev(case["lens"], torch)
    logits = torch.empty((1, cfg["vocab"]), dtype=torch.float16, device="cuda")
    m.decode_step(tok, tok, to_dev(case["bt"], torch), ld, logits=logits, use_graph=False)
    torch.cuda.synchronize()
    assert m.check_errors() == 0
    lens = case["lens"] + 1
    assert np.array_equal(to_host(ld), lens)
    x_in = case["embed"][case["tok"]]
    x_out = to_host(m.hidden(1))
    kp, vp = synth.host_pool(case, 0, "k"), synth.host_pool(case, 0, "v")
    check_layer_kernels(torch, orc, cfg, case["layers"][0], m, x_in, x_out, kp, vp, case["bt"], lens,
                        what="persistent step, layer 0")
    # the appended token: k rotated into place, v as projected (kp, vp now
    # hold the oracle's append of the device's q|k|v)
    pos = int(lens[0]) - 1
    page = int(case["bt"][0, pos // 16])
    assert_close(to_host(dls[0]["k_pool"])[page, :, pos % 16], kp[page, :, pos % 16], what="appended k")
    assert np.array_equal(to_host(dls[0]["v_pool"])[page, :, pos % 16], vp[page, :, pos % 16])
    # final norm + lm_head on the device's hidden state, then the argmax
    xn = orc.rmsnorm(x_out, case["fnorm"], cfg["eps"])
    ref = orc.fp16_gemv(xn[0], case["lm"])
    got = to_host(logits)[0]
    assert_close(got, ref, what="logits")
    err = float(np.max(np.abs(got.astype(np.float64) - ref)))
    srt = np.sort(ref)
    if srt[-1] - srt[-2] > 4 * err + 2e-3:
        assert int(to_host(tok)[0]) == orc.argmax(ref)
    m.close()


def test_persistent_one_qwen_layer_every_phase(api):
    """Qwen2.5-7B widths (hidden 3584, 28/4 heads, inter 18944, vocab
    152064), one layer, context 512: every phase of the step elementwise."""
    cfg = dict(synth.QWEN_MODEL, n_layers=1)
    case = synth.model_case(cfg, lens=[cfg["context"]], gen_tokens=4, pool_pages=64, seed=7100)
    _one_layer_every_phase(api, case, cfg["context"] + 16)


@pytest.mark.parametrize("cached", [0, 15, 16, 36, 63, 64, 127])
def test_persistent_tiny_layer_page_and_partition_boundaries(api, cached):
    """The new token on the first, last and next slot of a page and of a
    64-token attention partition (the unit the kernel splits attention by)."""
    cfg = dict(synth.TINY_LAYER, n_layers=1, vocab=1000, bias=True, codes="symmetric")
    case = synth.model_case(cfg, lens=[cached], gen_tokens=4, pool_pages=32, seed=7200 + cached)
    _one_layer_every_phase(api, case, 200)


def _tiny(n_layers, seed, lens=37, vocab=2000):
    cfg = dict(synth.TINY_LAYER, n_layers=n_layers, vocab=vocab, bias=True, codes="symmetric")
    return synth.model_case(cfg, lens=[lens], gen_tokens=24, pool_pages=32, seed=seed)


def test_persistent_free_running_matches_oracle(api):
    case = _tiny(3, 7300)
    cfg = case["cfg"]
    m, _ = _model(api, case, 128)
    tok = to_dev(case["tok"], torch)
    ld = to_dev(case["lens"], torch)
    btd = to_dev(case["bt"], torch)
    logits = torch.empty((1, cfg["vocab"]), dtype=torch.float16, device="cuda")
    kps = [synth.host_pool(case, l, "k") for l in range(cfg["n_layers"])]
    vps = [synth.host_pool(case, l, "v") for l in range(cfg["n_layers"])]
    t_or, n = case["tok"].copy(), case["lens"].copy()
    for step in range(12):
        m.decode_step(tok, tok, btd, ld, logits=logits, use_graph=True)
        n = n + 1
        t_next, lg_ref, _ = orc.decode_step(cfg, case["layers"], kps, vps, case["embed"], case["fnorm"], case["lm"],
                                            t_or, case["bt"], n, want_logits=True)
        got = to_host(logits)[0].astype(np.float64)
        ref = lg_ref[0].astype(np.float64)
        rel = np.sqrt(np.mean((got - ref) ** 2) / np.mean(ref ** 2))
        assert rel < 0.02, f"step {step}: logits differ by {rel:.3g} of their RMS"
        err = float(np.max(np.abs(got - ref)))
        srt = np.sort(ref)
        got_tok = int(to_host(tok)[0])
        if srt[-1] - srt[-2] > 4 * err + 2e-3:
            assert got_tok == int(t_next[0]), f"step {step}"
        elif got_tok != int(t_next[0]):
            break  # near-tie: the sequences may part here
        t_or = t_next
    assert m.check_errors() == 0
    m.close()


def test_persistent_agrees_with_kernel_path(api):
    """Same model, same start, both paths for 8 steps: the logits agree to
    the fp16 bound at every step while the tokens agree (the paths sum in
    different orders, so they are not bit-identical)."""
    case = _tiny(2, 7400)
    cfg = case["cfg"]
    runs = {}
    for path in ("kernels", "persistent"):
        m, _ = _model(api, case, 128, path=path)
        assert m.decode_path(1) == path
        tok = to_dev(case["tok"], torch)
        ld = to_dev(case["lens"], torch)
        btd = to_dev(case["bt"], torch)
        logits = torch.empty((1, cfg["vocab"]), dtype=torch.float16, device="cuda")
        seq = []
        for _ in range(8):
            m.decode_step(tok, tok, btd, ld, logits=logits, use_graph=True)
            seq.append((int(to_host(tok)[0]), to_host(logits)[0].astype(np.float64)))
        assert m.check_errors() == 0
        runs[path] = seq
        m.close()
    for step, ((tk, lk), (tp, lp)) in enumerate(zip(runs["kernels"], runs["persistent"])):
        rel = np.sqrt(np.mean((lk - lp) ** 2) / np.mean(lk ** 2))
        assert rel < 0.01, f"step {step}: paths differ by {rel:.3g} of the logits' RMS"
        if tk != tp:
            srt = np.sort(lk)
            assert srt[-1] - srt[-2] < 4 * float(np.max(np.abs(lk - lp))) + 2e-3, f"step {step}: tokens differ"
            break


def test_persistent_graph_replay_equals_direct_launch(api):
    case = _tiny(2, 7500)
    outs = []
    for use_graph in (False, True):
        m, dls = _model(api, case, 128)
        tok = to_dev(case["tok"], torch)
        ld = to_dev(case["lens"], torch)
        btd = to_dev(case["bt"], torch)
        logits = torch.empty((1, case["cfg"]["vocab"]), dtype=torch.float16, device="cuda")
        seq, lg = [], []
        for _ in range(5):
            m.decode_step(tok, tok, btd, ld, logits=logits, use_graph=use_graph)
            seq.append(int(to_host(tok)[0]))
            lg.append(to_host(logits).copy())
        outs.append((seq, lg, [to_host(d["k_pool"]) for d in dls]))
        m.close()
    (s0, l0, k0), (s1, l1, k1) = outs
    assert s0 == s1
    assert all(np.array_equal(a, b) for a, b in zip(l0, l1))   # the sums have a fixed order
    assert all(np.array_equal(a, b) for a, b in zip(k0, k1))


def test_persistent_barrier_abort_path_then_clean_step(api):
    """With the test hook's wait limit of 0 the first grid barrier that is
    not already complete gives up: every CTA leaves at its next barrier, the
    model reports W4A16_ERR_TIMEOUT and resets the kernel's counters, and the
    next step with the normal limit matches the oracle.  No barrier is left
    waiting on a CTA that never comes."""
    from w4a16_decode_paged_gb300 import _lib
    lib = _lib.load()
    case = _tiny(1, 7600, vocab=1000)
    cfg = case["cfg"]
    m, _ = _model(api, case, 128)
    btd = to_dev(case["bt"], torch)
    logits = torch.empty((1, cfg["vocab"]), dtype=torch.float16, device="cuda")
    old = lib.w4a16_debug_set_wait_limit_ns(0)
    try:
        tok = to_dev(case["tok"], torch)
        ld = to_dev(case["lens"], torch)
        m.decode_step(tok, tok, btd, ld, logits=logits, use_graph=False)
        assert m.check_errors() == 7      # W4A16_ERR_TIMEOUT
    finally:
        lib.w4a16_debug_set_wait_limit_ns(old)
    tok = to_dev(case["tok"], torch)
    ld = to_dev(case["lens"], torch)
    m.decode_step(tok, tok, btd, ld, logits=logits, use_graph=False)
    assert m.check_errors() == 0
    t_next, lg_ref, _ = orc.decode_step(cfg, case["layers"], [synth.host_pool(case, 0, "k")],
                                        [synth.host_pool(case, 0, "v")], case["embed"], case["fnorm"], case["lm"],
                                        case["tok"], case["bt"], case["lens"] + 1, want_logits=True)
    assert_close(to_host(logits), lg_ref, what="logits after the reset")
    m.close()


def test_persistent_reports_bad_page_and_skips_it(api):
    case = _tiny(1, 7700, vocab=500)
    bt = case["bt"].copy()
    pos = int(case["lens"][0])
    bt[0, pos // 16] = 10 ** 6                 # the page the new token lands in
    m, dls = _model(api, case, 128)
    tok = to_dev(case["tok"], torch)
    v_before = to_host(dls[0]["v_pool"]).copy()
    m.decode_step(tok, tok, to_dev(bt, torch), to_dev(case["lens"], torch), use_graph=False)
    assert m.check_errors() == 6               # W4A16_ERR_DEVICE_BOUNDS
    assert np.array_equal(to_host(dls[0]["v_pool"]), v_before)
    m.close()


def test_decode_path_selection(api):
    case = _tiny(1, 7800, vocab=500)
    m, _ = _model(api, case, 128, path="kernels")
    assert m.decode_path(1) == "kernels" and m.kernel_count(1) == 1 + 5 + 1
    m.set_decode_path("persistent")
    assert m.decode_path(1) == "persistent" and m.kernel_count(1) == 1
    m.set_decode_path("auto")
    assert m.decode_path(1) in ("kernels", "persistent")
    assert m.decode_path(2) == "kernels"
    m.close()
    # a model the persistent kernel does not cover (context beyond its merge)
    m, _ = _model(api, case, 8192, path="auto")
    assert m.decode_path(1) == "kernels"
    with pytest.raises(Exception):
        m.set_decode_path("persistent")
    m.close()
