"""The C-ABI library loads and exports every symbol include/*.h declares, and
its host-side argument checks reject bad calls before touching the GPU.
CPU only: no call here reaches a kernel launch."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from w4a16_decode_paged_gb300 import build
    build.build()
    from w4a16_decode_paged_gb300 import _lib
    return _lib.load()


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        for m in re.finditer(r"W4A16_API\s+[\w\s\*]+?\b(\w+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_header_declares_the_five_path_calls():
    names = _declared_symbols()
    for n in ("w4a16_gemv", "paged_gqa_decode", "kv_append_rope", "rmsnorm", "decode_step"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_symbols()
    assert len(names) >= 20
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_signatures_cover_the_header(lib):
    from w4a16_decode_paged_gb300 import _lib
    assert _declared_symbols() <= set(_lib.SIGNATURES)


def test_version(lib):
    assert lib.w4a16_version() == 100


ALIGNED = 1 << 20          # fake device addresses: never dereferenced
MISALIGNED = (1 << 20) + 64


def test_gemv_rejects_bad_shapes_and_alignment(lib):
    from w4a16_decode_paged_gb300 import _lib
    rc = lib.w4a16_gemv(ALIGNED, 1, 100, ALIGNED, ALIGNED, 8, None, None, ALIGNED, None)
    assert rc == 3 and b"multiple of 128" in lib.w4a16_last_error()
    rc = lib.w4a16_gemv(MISALIGNED, 1, 128, ALIGNED, ALIGNED, 8, None, None, ALIGNED, None)
    assert rc == 2 and b"x must be 128-byte aligned" in lib.w4a16_last_error()
    rc = lib.w4a16_gemv(ALIGNED, 1, 128, ALIGNED, MISALIGNED, 8, None, None, ALIGNED, None)
    assert rc == 2
    rc = lib.w4a16_gemv(None, 1, 128, ALIGNED, ALIGNED, 8, None, None, ALIGNED, None)
    assert rc == 1
    rc = lib.w4a16_gemv(ALIGNED, 0, 128, ALIGNED, ALIGNED, 8, None, None, ALIGNED, None)
    assert rc == 1
    rc = lib.w4a16_gemv(ALIGNED, 64, 4096, ALIGNED, ALIGNED, 8, None, None, ALIGNED, None)
    assert rc == 3  # M = 64: above the largest batch (32)
    with pytest.raises(_lib.W4A16Error):
        _lib.check(rc)


def test_attention_rejects_bad_shapes(lib):
    args = lambda D=128, Hq=28, Hkv=4, part=512, ws=None, wsb=0, maxctx=512: (
        ALIGNED, 0, ALIGNED, ALIGNED, 64, ALIGNED, 32, ALIGNED, maxctx, 1, Hq, Hkv, D, 0.088, part, ws, wsb,
        ALIGNED, None, None)
    assert lib.paged_gqa_decode(*args(D=64)) == 3
    assert lib.paged_gqa_decode(*args(Hq=30, Hkv=4)) == 3
    assert lib.paged_gqa_decode(*args(Hq=36, Hkv=4)) == 3          # 9 heads per kv head
    assert lib.paged_gqa_decode(*args(part=100)) == 3
    assert lib.paged_gqa_decode(*args(maxctx=1024)) == 3           # beyond max_blocks * 16
    assert lib.paged_gqa_decode(*args(part=64)) == 1               # needs a workspace
    need = lib.paged_gqa_decode_workspace_size(1, 28, 4, 512, 64, 128)
    assert need >= 28 * 8 * 128 * 4
    assert lib.paged_gqa_decode(*args(part=64, ws=MISALIGNED, wsb=need)) == 2


def test_append_rejects_bad_shapes(lib):
    base = [ALIGNED, ALIGNED, ALIGNED, 0, ALIGNED, ALIGNED, 64, ALIGNED, 4, ALIGNED, 1, 28, 4, 128, 1e6, None, None]
    a = list(base); a[13] = 64
    assert lib.kv_append_rope(*a) == 3
    a = list(base); a[11] = 27
    assert lib.kv_append_rope(*a) == 3
    a = list(base); a[14] = 0.0
    assert lib.kv_append_rope(*a) == 1
    a = list(base); a[4] = MISALIGNED
    assert lib.kv_append_rope(*a) == 2


def test_rmsnorm_lm_head_reject(lib):
    assert lib.rmsnorm(ALIGNED, ALIGNED, ALIGNED, 1, 12, 1e-6, None) == 3
    assert lib.rmsnorm(ALIGNED, ALIGNED, MISALIGNED, 1, 16, 1e-6, None) == 2
    ws = lib.lm_head_argmax_workspace_size(1, 1000)
    assert lib.lm_head_argmax(ALIGNED, 5, 896, ALIGNED, 1000, None, ALIGNED, ALIGNED, ws, None) == 3
    assert lib.lm_head_argmax(ALIGNED, 1, 896, ALIGNED, 1000, None, ALIGNED, ALIGNED, 8, None) == 1


def test_model_create_rejects_bad_config(lib):
    from w4a16_decode_paged_gb300 import _lib
    c = _lib.ModelConfig(896, 7, 1, 64, 2432, 1, 0, 1e-6, 1e6, 8, 0)
    w = _lib.ModelWeights(None, None, None, None)
    h = ctypes.c_void_p()
    assert lib.w4a16_model_create(ctypes.byref(c), ctypes.byref(w), 1, 64, ctypes.byref(h)) == 3
    c = _lib.ModelConfig(896, 7, 1, 128, 2432, 1, 0, 1e-6, 1e6, 8, 0)
    assert lib.w4a16_model_create(ctypes.byref(c), ctypes.byref(w), 1, 64, ctypes.byref(h)) == 1
    assert not h.value


def test_tensor_core_calls_reject(lib):
    # w4a16_gemm(x, M, K, qweight, scales, N, bias, residual, y, workspace, bytes, stream)
    good = [ALIGNED, 8, 256, ALIGNED, ALIGNED, 128, None, None, ALIGNED, None, 0, None]
    for i, v, rc in ((1, 129, 3), (2, 200, 3), (0, None, 1), (3, None, 1), (0, MISALIGNED, 2),
                     (8, MISALIGNED, 2), (9, MISALIGNED, 2), (7, MISALIGNED, 2), (1, 0, 1)):
        a = list(good); a[i] = v
        assert lib.w4a16_gemm(*a) == rc, (i, v)
    # w4a16_gemm_silu_mul(x, M, K, qg, sg, qu, su, N, y, workspace, bytes, stream)
    good = [ALIGNED, 8, 256, ALIGNED, ALIGNED, ALIGNED, ALIGNED, 128, ALIGNED, None, 0, None]
    for i, v, rc in ((5, None, 1), (6, MISALIGNED, 2), (1, 65, 3), (2, 130, 3)):
        a = list(good); a[i] = v
        assert lib.w4a16_gemm_silu_mul(*a) == rc, (i, v)
    assert lib.w4a16_gemm_workspace_size(8, 64, 128, 0) == 0      # K below one scale group
    assert lib.w4a16_gemm_workspace_size(32, 18944, 3584, 0) > 8192  # split K: tickets + partial tiles
    assert lib.w4a16_gemm_workspace_size(128, 18944, 3584, 0) > 8192  # a prompt's row block: wider tiles
    # lm_head_logits_batched(x, B, H, lm_head, vocab, logits, stream)
    assert lib.lm_head_logits_batched(ALIGNED, 33, 896, ALIGNED, 1000, ALIGNED, None) == 3
    assert lib.lm_head_logits_batched(ALIGNED, 8, 900, ALIGNED, 1000, ALIGNED, None) == 3
    assert lib.lm_head_logits_batched(ALIGNED, 8, 896, ALIGNED, 1000, MISALIGNED, None) == 2
    assert lib.lm_head_logits_batched(ALIGNED, 8, 896, None, 1000, ALIGNED, None) == 1
    # argmax_rows(logits, B, vocab, tokens, logits16, stream)
    assert lib.argmax_rows(None, 2, 10, ALIGNED, None, None) == 1
    assert lib.argmax_rows(ALIGNED, 0, 10, ALIGNED, None, None) == 1


def test_fused_gemv_and_gather_calls_reject(lib):
    # w4a16_gemv_rmsnorm(x, gamma, eps, M, K, qweight, scales, N, bias, y, stream)
    good = [ALIGNED, ALIGNED, 1e-6, 1, 256, ALIGNED, ALIGNED, 64, None, ALIGNED, None]
    for i, v, rc in ((1, None, 1), (2, -1.0, 1), (4, 200, 3), (1, MISALIGNED, 2), (9, MISALIGNED, 2)):
        a = list(good); a[i] = v
        assert lib.w4a16_gemv_rmsnorm(*a) == rc, (i, v)
    # w4a16_gemv_silu_mul(x, gamma, eps, M, K, qg, sg, qu, su, N, y, stream)
    good = [ALIGNED, None, 1e-6, 1, 256, ALIGNED, ALIGNED, ALIGNED, ALIGNED, 64, ALIGNED, None]
    for i, v, rc in ((7, None, 1), (2, -1.0, 1), (5, MISALIGNED, 2), (4, 100, 3)):
        a = list(good); a[i] = v
        assert lib.w4a16_gemv_silu_mul(*a) == rc, (i, v)
    # embedding_gather(embed, vocab, H, tokens, B, x, err_flag, stream)
    assert lib.embedding_gather(ALIGNED, 100, 12, ALIGNED, 1, ALIGNED, None, None) == 3
    assert lib.embedding_gather(None, 100, 16, ALIGNED, 1, ALIGNED, None, None) == 1
    assert lib.embedding_gather(ALIGNED, 100, 16, ALIGNED, 0, ALIGNED, None, None) == 1
    assert lib.embedding_gather(MISALIGNED, 100, 16, ALIGNED, 1, ALIGNED, None, None) == 2


def test_model_calls_reject_a_null_model(lib):
    assert lib.decode_step(None, ALIGNED, ALIGNED, ALIGNED, 4, ALIGNED, 1, None, 1, None) == 1
    assert lib.w4a16_model_layer(None, 0, ALIGNED, ALIGNED, 4, ALIGNED, 1, None) == 1
    assert lib.w4a16_model_hidden(None, ALIGNED, 1, None) == 1
    assert lib.w4a16_model_activation(None, 0, ALIGNED, 1, None) == 1
    assert lib.w4a16_model_check_errors(None, None) == 1
    assert lib.decode_step_kernel_count(None, 1) == 0
    assert b"null" in lib.w4a16_last_error()


def test_default_partition_rule(lib):
    """Host-side choice of the attention partition (no GPU call)."""
    f = lib.paged_gqa_decode_default_partition
    assert f(1, 4, 512) == 128 and f(32, 4, 1024) == 128      # one cluster of 128-token partitions
    assert f(4, 4, 32768) == 512 and f(1, 4, 2000) == 512      # few (sequence, kv head) pairs
    assert f(32, 4, 4096) == 256 and f(16, 4, 1025) == 256     # many pairs: a warp per 256 tokens
    assert f(0, 4, 512) == 64                                  # invalid sizes: a fallback value


def test_attention_workspace_holds_every_partial(lib):
    """Host-side workspace size (no GPU call): room for each (sequence, q head,
    partition) partial -- 128 fp32 output dims plus its running max and sum --
    and it grows with the batch, the context and finer partitions."""
    f = lib.paged_gqa_decode_workspace_size
    for B, Hq, Hkv, L, part in ((1, 28, 4, 512, 128), (4, 28, 4, 32768, 512), (32, 28, 4, 4096, 256),
                                (3, 8, 8, 1000, 64), (2, 28, 4, 17, 16)):
        P = -(-L // part)
        ws = f(B, Hq, Hkv, L, part, 128)
        assert ws >= B * Hq * P * (128 + 2) * 4, (B, L, part)
        assert ws % 128 == 0
        assert f(B + 1, Hq, Hkv, L, part, 128) >= ws
        assert f(B, Hq, Hkv, 2 * L, part, 128) >= ws
        if part >= 32:
            assert f(B, Hq, Hkv, L, part // 2, 128) >= ws
