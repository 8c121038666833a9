"""The torch binding's argument checks and marshalling, on the CPU.

The library only sees pointers and sizes, so the binding is where a wrong
extent, dtype or layout has to be caught before it becomes an out-of-bounds
access on the GPU.  Here the library is replaced by a recorder and the
device check by a stub, so every binding runs on CPU tensors: valid calls
(the shapes the tests and the benchmark use) must reach the library with
the right sizes, invalid ones must raise ValueError naming the argument."""
import pytest

torch = pytest.importorskip("torch")

from w4a16_decode_paged_gb300 import api  # noqa: E402


class _Recorder:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def fn(*args):
            self.calls.append((name, args))
            return 0
        return fn


@pytest.fixture
def lib(monkeypatch):
    rec = _Recorder()
    monkeypatch.setattr(api, "load", lambda: rec)
    monkeypatch.setattr(api, "_on_device", lambda t: True)
    monkeypatch.setattr(api, "stream_handle", lambda stream=None: 0)
    return rec


def h(*shape):
    return torch.zeros(shape, dtype=torch.float16)


def i32(*shape):
    return torch.zeros(shape, dtype=torch.int32)


def last(lib, name):
    calls = [a for n, a in lib.calls if n == name]
    assert calls, f"{name} not called"
    return calls[-1]


def test_gemv_reaches_the_library_with_its_sizes(lib):
    M, K, N = 3, 256, 40
    y = api.w4a16_gemv(h(M, K), i32(N, K // 8), h(N, K // 128), bias=h(N), residual=h(M, N))
    assert tuple(y.shape) == (M, N) and y.dtype == torch.float16
    a = last(lib, "w4a16_gemv")
    assert (a[1], a[2], a[5]) == (M, K, N)
    api.w4a16_gemv(h(M, K), torch.zeros((N, K // 8), dtype=torch.uint32), h(N, K // 128), out=h(M, N))


@pytest.mark.parametrize("bad,what", [
    (dict(scales=h(40, 3)), "scales"),
    (dict(qweight=i32(40, 31)), "qweight"),
    (dict(bias=h(39)), "bias"),
    (dict(residual=h(2, 40)), "residual"),
    (dict(out=h(3, 41)), "out"),
    (dict(x=h(256)), "x"),
    (dict(x=torch.zeros((3, 256), dtype=torch.float32)), "x"),
    (dict(x=h(256, 3).t()), "x"),
    (dict(qweight=torch.zeros((40, 32), dtype=torch.int64)), "qweight"),
])
def test_gemv_rejects_what_would_be_read_out_of_bounds(lib, bad, what):
    args = dict(x=h(3, 256), qweight=i32(40, 32), scales=h(40, 2), bias=None, residual=None, out=None)
    args.update(bad)
    with pytest.raises(ValueError, match=what):
        api.w4a16_gemv(**args)
    assert not lib.calls


def test_tensor_core_gemm_and_silu_checks(lib):
    M, K, N = 8, 384, 130
    api.w4a16_gemm(h(M, K), i32(N, K // 8), h(N, K // 128), residual=h(M, N), workspace=torch.zeros(256, dtype=torch.uint8))
    with pytest.raises(ValueError, match="workspace"):
        api.w4a16_gemm(h(M, K), i32(N, K // 8), h(N, K // 128), workspace=torch.zeros(64, dtype=torch.float32))
    y = api.w4a16_gemm_silu_mul(h(M, K), i32(N, K // 8), h(N, K // 128), i32(N, K // 8), h(N, K // 128))
    assert tuple(y.shape) == (M, N)
    with pytest.raises(ValueError, match="qweight_up"):
        api.w4a16_gemm_silu_mul(h(M, K), i32(N, K // 8), h(N, K // 128), i32(N + 2, K // 8), h(N + 2, K // 128))
    with pytest.raises(ValueError, match="scales_up"):
        api.w4a16_gemm_silu_mul(h(M, K), i32(N, K // 8), h(N, K // 128), i32(N, K // 8), h(N, K // 64))


def test_fused_norm_bindings(lib):
    M, K, N = 2, 3584, 64
    api.w4a16_gemv_rmsnorm(h(M, K), h(K), 1e-6, i32(N, K // 8), h(N, K // 128), bias=h(N))
    with pytest.raises(ValueError, match="gamma"):
        api.w4a16_gemv_rmsnorm(h(M, K), h(K - 128), 1e-6, i32(N, K // 8), h(N, K // 128))
    api.w4a16_gemv_silu_mul(h(M, K), None, 1e-6, i32(N, K // 8), h(N, K // 128), i32(N, K // 8), h(N, K // 128))
    a = last(lib, "w4a16_gemv_silu_mul")
    assert a[1] is None and (a[3], a[4], a[9]) == (M, K, N)
    with pytest.raises(ValueError, match="gamma"):
        api.w4a16_gemv_silu_mul(h(M, K), h(1), 1e-6, i32(N, K // 8), h(N, K // 128), i32(N, K // 8), h(N, K // 128))
    y = api.rmsnorm(h(M, K), h(K), 1e-6)
    assert tuple(y.shape) == (M, K)
    with pytest.raises(ValueError, match="out"):
        api.rmsnorm(h(M, K), h(K), 1e-6, out=h(M, K + 8))


def test_lm_head_and_argmax_bindings(lib):
    B, H, V = 3, 896, 4099
    toks, logits = api.lm_head_argmax(h(B, H), h(V, H), want_logits=True)
    assert tuple(toks.shape) == (B,) and tuple(logits.shape) == (B, V)
    with pytest.raises(ValueError, match="lm_head"):
        api.lm_head_argmax(h(B, H), h(V, H + 1))
    with pytest.raises(ValueError, match="tokens_out"):
        api.lm_head_argmax(h(B, H), h(V, H), tokens_out=i32(B + 1))
    lg = api.lm_head_logits_batched(h(B, H), h(V, H))
    assert lg.dtype == torch.float32 and tuple(lg.shape) == (B, V)
    with pytest.raises(ValueError, match="out"):
        api.lm_head_logits_batched(h(B, H), h(V, H), out=h(B, V))
    api.argmax_rows(torch.zeros((B, V)), logits16=h(B, V))
    with pytest.raises(ValueError, match="logits16"):
        api.argmax_rows(torch.zeros((B, V)), logits16=h(B, V - 1))
    x = api.embedding_gather(h(300, 896), i32(4))
    assert tuple(x.shape) == (4, 896)
    with pytest.raises(ValueError, match="tokens"):
        api.embedding_gather(h(300, 896), torch.zeros(4, dtype=torch.int64))


def test_attention_bindings(lib):
    B, Hq, Hkv, D, pages = 2, 28, 4, 128, 40
    kp, vp = h(pages, Hkv, 16, D), h(pages, Hkv, 16, D)
    bt, lens = i32(B, 19), i32(B)
    out = api.paged_gqa_decode(h(B, Hq, D), kp, vp, bt, lens, max_context=300, partition_tokens=64)
    assert tuple(out.shape) == (B, Hq, D)
    a = last(lib, "paged_gqa_decode")
    assert (a[4], a[6], a[9], a[10], a[11], a[12]) == (pages, 19, B, Hq, Hkv, D)
    row = h(B, (Hq + 2 * Hkv) * D)
    api.paged_gqa_decode(row, kp, vp, bt, lens, max_context=300, q_stride=row.shape[1], n_q_heads=Hq)
    with pytest.raises(ValueError, match="q"):
        api.paged_gqa_decode(h(B - 1, Hq, D), kp, vp, bt, lens, max_context=300)
    with pytest.raises(ValueError, match="k_pool"):
        api.paged_gqa_decode(h(B, Hq, D), h(pages, Hkv, 8, D), vp, bt, lens, max_context=300)
    with pytest.raises(ValueError, match="v_pool"):
        api.paged_gqa_decode(h(B, Hq, D), kp, h(pages - 1, Hkv, 16, D), bt, lens, max_context=300)
    with pytest.raises(ValueError, match="context_lens"):
        api.paged_gqa_decode(h(B, Hq, D), kp, vp, bt, i32(B + 1), max_context=300)
    with pytest.raises(ValueError, match="block_table"):
        api.paged_gqa_decode(h(B, Hq, D), kp, vp, i32(B * 19), lens, max_context=300)
    out = api.paged_gqa_decode_rope_append(row, kp, vp, bt, lens, max_context=300, theta=1e6, n_q_heads=Hq)
    assert tuple(out.shape) == (B, Hq, D)
    with pytest.raises(ValueError, match="qkv"):
        api.paged_gqa_decode_rope_append(h(B, Hq * D), kp, vp, bt, lens, max_context=300, theta=1e6, n_q_heads=Hq)
    api.kv_append_rope(h(B, Hq, D), h(B, Hkv, D), h(B, Hkv, D), kp, vp, bt, lens, 1e6, err_flag=i32(1))
    with pytest.raises(ValueError, match="err_flag"):
        api.kv_append_rope(h(B, Hq, D), h(B, Hkv, D), h(B, Hkv, D), kp, vp, bt, lens, 1e6, err_flag=h(1))


def test_host_tensors_are_refused(monkeypatch):
    monkeypatch.setattr(api, "load", lambda: _Recorder())
    with pytest.raises(ValueError, match="CUDA"):
        api.w4a16_gemv(h(1, 128), i32(8, 16), h(8, 1))


def _tiny_model(lib):
    cfg = dict(hidden=128, n_q_heads=7, n_kv_heads=1, head_dim=128, inter=256, vocab=50, eps=1e-6, theta=1e6)
    pool = h(8, 1, 16, 128)
    layer = {k: h(1) for k in api.Model.LAYER_KEYS}
    layer.update(k_pool=pool, v_pool=pool)
    return api.Model(cfg, [layer], embed=h(50, 128), final_norm=h(128), lm_head=h(50, 128), max_batch=2,
                     max_context=64, num_pages=8)


def test_model_step_and_layer_arguments(lib):
    m = _tiny_model(lib)
    tok, bt, lens = i32(2), i32(2, 4), i32(2)
    m.decode_step(tok, tok, bt, lens, logits=h(2, 50))
    a = last(lib, "decode_step")
    assert (a[4], a[6]) == (4, 2)                     # max_blocks, B
    with pytest.raises(ValueError, match="logits"):
        m.decode_step(tok, tok, bt, lens, logits=h(2, 49))
    with pytest.raises(ValueError, match="context_lens"):
        m.decode_step(tok, tok, bt, i32(1))
    with pytest.raises(ValueError, match="block_table"):
        m.decode_step(tok, tok, i32(1, 4), lens)
    with pytest.raises(ValueError, match="tokens_out"):
        m.decode_step(tok, i32(3), bt, lens)
    with pytest.raises(ValueError, match="tokens_in"):
        m.decode_step(torch.zeros(2, dtype=torch.int64), tok, bt, lens)
    m.layer(0, h(2, 128), bt, lens)
    with pytest.raises(ValueError, match="x"):
        m.layer(0, h(2, 64), bt, lens)
    m.close()
