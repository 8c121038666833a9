"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
import numpy as np

# fp16 outputs: |got - ref| <= ATOL + RTOL * |ref| elementwise, ref = oracle (fp64, one fp16 rounding)
ATOL = 1e-2
RTOL = 2e-3


def to_dev(a, torch):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).cuda()


def to_host(t):
    return t.detach().cpu().numpy()


def assert_close(got, ref, atol=ATOL, rtol=RTOL, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"got {got[i]} ref {ref[i]} (err {err[i]:.3g}, bound {bound[i]:.3g})")


def max_rel(got, ref, floor=1e-2):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    m = np.abs(ref) > floor
    return float(np.max(np.abs(got[m] - ref[m]) / np.abs(ref[m]))) if m.any() else 0.0


def assert_rms_close(got, ref, rtol=RTOL, what=""):
    """Composite outputs (several fp16-rounded kernels chained): the RMS of
    the error within rtol of the RMS of the output.  Each kernel on the way
    is held to the elementwise bound on its own inputs separately."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rel = np.sqrt(np.mean((got - ref) ** 2) / np.mean(ref ** 2))
    assert rel <= rtol, f"{what}: RMS error {rel:.3g} of the output RMS (bound {rtol})"


def check_layer_kernels(torch, orc, cfg, w, model, x_in, x_out, k_pool, v_pool, block_table, context_lens,
                        rows=None, what=""):
    """Each kernel of one decoder layer, held to the elementwise fp16 bound on
    its own device inputs (read back from the model's arena after
    model.layer): RMSNorm + q|k|v projection on x_in; RoPE + KV append +
    paged attention on the device's q|k|v (k_pool / v_pool: host copies of
    the pools before the layer, appended in place here); o projection +
    residual on the device's attention output; RMSNorm + gate/up + SiLU-mul
    on the device's post-attention state; down projection + residual on the
    device's MLP activations.  `rows` picks the sequences checked."""
    B = x_in.shape[0]
    rows = list(range(B)) if rows is None else list(rows)
    H, Hq, Hkv, D = cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    eps, theta = cfg["eps"], cfg["theta"]
    qkv = to_host(model.activation("qkv", B))[rows]
    att = to_host(model.activation("attn", B))[rows]
    h = to_host(model.activation("resid", B))[rows]
    mlp = to_host(model.activation("mlp", B))[rows]
    xi, xo = np.asarray(x_in)[rows], np.asarray(x_out)[rows]
    bt, lens = np.asarray(block_table)[rows], np.asarray(context_lens)[rows]
    n = len(rows)

    xn = orc.rmsnorm(xi, w["ln1"], eps)
    ref = np.concatenate([orc.w4a16_gemv(xn, w["w" + p], w["s" + p], bias=w.get("b" + p)) for p in "qkv"], axis=1)
    assert_close(qkv, ref, what=f"{what} rmsnorm + q|k|v")

    qd = qkv[:, :Hq * D].reshape(n, Hq, D)
    kd = qkv[:, Hq * D:(Hq + Hkv) * D].reshape(n, Hkv, D)
    vd = qkv[:, (Hq + Hkv) * D:].reshape(n, Hkv, D)
    q_rot = np.stack([orc.rope(qd[i], int(lens[i]) - 1, theta) for i in range(n)])
    k_rot = np.stack([orc.rope(kd[i], int(lens[i]) - 1, theta) for i in range(n)])
    orc.kv_append(k_rot, vd, k_pool, v_pool, bt, lens)
    ref = orc.paged_attention(q_rot, k_pool, v_pool, bt, lens, 1.0 / np.sqrt(D)).reshape(n, Hq * D)
    assert_close(att, ref, what=f"{what} rope + append + attention")

    assert_close(h, orc.w4a16_gemv(att, w["wo"], w["so"], residual=xi), what=f"{what} o + residual")

    hn = orc.rmsnorm(h, w["ln2"], eps)
    ref = orc.silu_mul(orc.w4a16_gemv(hn, w["wg"], w["sg"]), orc.w4a16_gemv(hn, w["wu"], w["su"]))
    assert_close(mlp, ref, what=f"{what} rmsnorm + gate|up + silu-mul")

    assert_close(xo, orc.w4a16_gemv(mlp, w["wd"], w["sd"], residual=h), what=f"{what} down + residual")


def layer_parity(api, torch, orc, synth, cfg, lens=None, seed=None, partition_tokens=0):
    """One decoder layer through the model handle: every kernel on its own
    device inputs (check_layer_kernels), the pools (only the appended slots
    change, placement bit-exact, values to the fp16 bound), the layer output
    against the oracle's whole layer (RMS bound) and the device error word."""
    case = synth.layer_case(cfg, lens=lens, seed=seed)
    w = case["weights"]
    dl = api.device_layer(w, case["k_pool"], case["v_pool"])
    model = api.Model(cfg, [dl], max_batch=cfg["batch"], max_context=int(case["context_lens"].max()) + 16,
                      num_pages=case["k_pool"].shape[0], partition_tokens=partition_tokens)
    x = to_dev(case["x"], torch)
    bt = to_dev(case["block_table"], torch)
    ld = to_dev(case["context_lens"], torch)
    model.layer(0, x, bt, ld)
    torch.cuda.synchronize()
    x_out = to_host(x)
    kp, vp = case["k_pool"].copy(), case["v_pool"].copy()
    check_layer_kernels(torch, orc, cfg, w, model, case["x"], x_out, kp, vp, case["block_table"],
                        case["context_lens"], what=cfg["name"])
    # pools: only the appended slots changed (placement bit-exact); values to
    # the fp16 bound against the oracle's rotation of the device's k
    appended = {(int(case["block_table"][b, (L - 1) // 16]), (L - 1) % 16) for b, L in enumerate(case["context_lens"])}
    pages = sorted({p for p, _ in appended})
    for name, ref_pool in (("k_pool", kp), ("v_pool", vp)):
        got = to_host(dl[name])
        diff = np.any(got != case[name], axis=-1)
        for pg, h, sl in np.argwhere(diff):
            assert (int(pg), int(sl)) in appended, (name, pg, h, sl)
        assert_close(got[pages], ref_pool[pages], what=name)
    # the whole layer against the oracle's own chain
    kp, vp = case["k_pool"].copy(), case["v_pool"].copy()
    ref = orc.decoder_layer(cfg, w, case["x"], kp, vp, case["block_table"], case["context_lens"])
    assert_rms_close(x_out, ref, what=f"{cfg['name']} layer output")
    assert model.check_errors() == 0
    model.close()
