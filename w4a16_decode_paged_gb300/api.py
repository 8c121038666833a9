"""Torch-tensor front end of the C ABI (same names as include/w4a16.h).

Each function checks dtypes/devices, allocates outputs with torch when the
caller gives none, and calls the library on torch's current CUDA stream.
Nothing here computes any part of the decode path.
"""
from __future__ import annotations

import ctypes
import math

import torch

from ._lib import LayerWeights, ModelConfig, ModelWeights, check, load

__all__ = ["w4a16_gemv", "w4a16_gemm", "w4a16_gemm_silu_mul", "lm_head_logits_batched", "argmax_rows", "w4a16_gemv_rmsnorm", "w4a16_gemv_silu_mul", "rmsnorm", "kv_append_rope",
           "paged_gqa_decode", "paged_gqa_decode_rope_append", "paged_gqa_decode_workspace_size", "paged_gqa_decode_default_partition",
           "workspace_clear", "embedding_gather", "lm_head_argmax", "Model", "stream_handle"]


def stream_handle(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _p(t):
    return None if t is None else t.data_ptr()


def _on_device(t) -> bool:
    return t.is_cuda


def _arg(t, dtypes, name, shape=None, optional=False):
    """Check one tensor argument before its pointer goes to the library:
    dtype, contiguity, shape (entries None match any extent) and device.
    The library only sees pointers and sizes, so a wrong extent here would
    become an out-of-bounds access on the GPU."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and (t.dim() != len(shape) or
                              any(e is not None and t.shape[i] != e for i, e in enumerate(shape))):
        want = tuple("*" if e is None else e for e in shape)
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {want}")
    if not _on_device(t):
        raise ValueError(f"{name} must be a CUDA tensor")


_H = (torch.float16,)
_W = (torch.int32, torch.uint32)
_I = (torch.int32,)
_F = (torch.float32,)
_U8 = (torch.uint8,)


def _xk(x):
    """(M, K) of the activations x [M][K] (fp16)."""
    _arg(x, _H, "x")
    if x.dim() != 2:
        raise ValueError(f"x: shape {tuple(x.shape)}, expected (M, K)")
    return x.shape[0], x.shape[1]


def _paging(k_pool, v_pool, block_table, context_lens):
    """(pages, Hkv, D, B) of pools [pages][Hkv][16][D], a block table
    [B][max_blocks] and context_lens [B]."""
    _arg(k_pool, _H, "k_pool", (None, None, 16, None))
    pages, Hkv, _, D = k_pool.shape
    _arg(v_pool, _H, "v_pool", tuple(k_pool.shape))
    _arg(block_table, _I, "block_table", (None, None))
    B = block_table.shape[0]
    _arg(context_lens, _I, "context_lens", (B,))
    return pages, Hkv, D, B


def _int4(qweight, scales, K, name="qweight", sname="scales"):
    """N of a packed int4 matrix qweight [N][K/8] with scales [N][K/128]."""
    _arg(qweight, _W, name)
    if qweight.dim() != 2:
        raise ValueError(f"{name}: shape {tuple(qweight.shape)}, expected (N, {K // 8})")
    N = qweight.shape[0]
    _arg(qweight, _W, name, (N, K // 8))
    _arg(scales, _H, sname, (N, K // 128))
    return N


def w4a16_gemv(x, qweight, scales, bias=None, residual=None, out=None, stream=None):
    M, K = _xk(x)
    N = _int4(qweight, scales, K)
    _arg(bias, _H, "bias", (N,), optional=True)
    _arg(residual, _H, "residual", (M, N), optional=True)
    _arg(out, _H, "out", (M, N), optional=True)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    check(load().w4a16_gemv(_p(x), M, K, _p(qweight), _p(scales), N, _p(bias), _p(residual), _p(out),
                            stream_handle(stream)))
    return out


def w4a16_gemm(x, qweight, scales, bias=None, residual=None, out=None, workspace=None, split=True, stream=None):
    """Tensor-core path for a batch of rows: decode batches (M <= 32) and the
    wider row blocks of a prompt (M <= 128)."""
    M, K = _xk(x)
    N = _int4(qweight, scales, K)
    _arg(bias, _H, "bias", (N,), optional=True)
    _arg(residual, _H, "residual", (M, N), optional=True)
    _arg(out, _H, "out", (M, N), optional=True)
    _arg(workspace, _U8, "workspace", optional=True)
    lib = load()
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    if workspace is None and split:
        workspace = torch.zeros(max(256, lib.w4a16_gemm_workspace_size(M, K, N, 0)), dtype=torch.uint8,
                                device=x.device)
    check(lib.w4a16_gemm(_p(x), M, K, _p(qweight), _p(scales), N, _p(bias), _p(residual), _p(out), _p(workspace),
                         0 if workspace is None else workspace.numel(), stream_handle(stream)))
    return out


def w4a16_gemm_silu_mul(x, qweight_gate, scales_gate, qweight_up, scales_up, out=None, workspace=None, split=True,
                        stream=None):
    M, K = _xk(x)
    N = _int4(qweight_gate, scales_gate, K, "qweight_gate", "scales_gate")
    _int4(qweight_up, scales_up, K, "qweight_up", "scales_up")
    if qweight_up.shape[0] != N:
        raise ValueError(f"qweight_up: {qweight_up.shape[0]} rows, qweight_gate {N}")
    _arg(out, _H, "out", (M, N), optional=True)
    _arg(workspace, _U8, "workspace", optional=True)
    lib = load()
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    if workspace is None and split:
        workspace = torch.zeros(max(256, lib.w4a16_gemm_workspace_size(M, K, N, 1)), dtype=torch.uint8,
                                device=x.device)
    check(lib.w4a16_gemm_silu_mul(_p(x), M, K, _p(qweight_gate), _p(scales_gate), _p(qweight_up), _p(scales_up), N,
                                  _p(out), _p(workspace), 0 if workspace is None else workspace.numel(),
                                  stream_handle(stream)))
    return out


def lm_head_logits_batched(x, lm_head, out=None, stream=None):
    B, H = _xk(x)
    _arg(lm_head, _H, "lm_head", (None, H))
    V = lm_head.shape[0]
    _arg(out, _F, "out", (B, V), optional=True)
    if out is None:
        out = torch.empty((B, V), dtype=torch.float32, device=x.device)
    check(load().lm_head_logits_batched(_p(x), B, H, _p(lm_head), V, _p(out), stream_handle(stream)))
    return out


def argmax_rows(logits32, tokens_out=None, logits16=None, stream=None):
    _arg(logits32, _F, "logits32", (None, None))
    B, V = logits32.shape
    _arg(tokens_out, _I, "tokens_out", (B,), optional=True)
    _arg(logits16, _H, "logits16", (B, V), optional=True)
    if tokens_out is None:
        tokens_out = torch.empty(B, dtype=torch.int32, device=logits32.device)
    check(load().argmax_rows(_p(logits32), B, V, _p(tokens_out), _p(logits16), stream_handle(stream)))
    return tokens_out


def w4a16_gemv_rmsnorm(x, gamma, eps, qweight, scales, bias=None, out=None, stream=None):
    M, K = _xk(x)
    _arg(gamma, _H, "gamma", (K,))
    N = _int4(qweight, scales, K)
    _arg(bias, _H, "bias", (N,), optional=True)
    _arg(out, _H, "out", (M, N), optional=True)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    check(load().w4a16_gemv_rmsnorm(_p(x), _p(gamma), float(eps), M, K, _p(qweight), _p(scales), N, _p(bias),
                                    _p(out), stream_handle(stream)))
    return out


def w4a16_gemv_silu_mul(x, gamma, eps, qweight_gate, scales_gate, qweight_up, scales_up, out=None, stream=None):
    M, K = _xk(x)
    _arg(gamma, _H, "gamma", (K,), optional=True)
    N = _int4(qweight_gate, scales_gate, K, "qweight_gate", "scales_gate")
    _int4(qweight_up, scales_up, K, "qweight_up", "scales_up")
    if qweight_up.shape[0] != N:
        raise ValueError(f"qweight_up: {qweight_up.shape[0]} rows, qweight_gate {N}")
    _arg(out, _H, "out", (M, N), optional=True)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    check(load().w4a16_gemv_silu_mul(_p(x), _p(gamma), float(eps), M, K, _p(qweight_gate), _p(scales_gate),
                                     _p(qweight_up), _p(scales_up), N, _p(out), stream_handle(stream)))
    return out


def rmsnorm(x, gamma, eps, out=None, stream=None):
    M, H = _xk(x)
    _arg(gamma, _H, "gamma", (H,))
    _arg(out, _H, "out", (M, H), optional=True)
    if out is None:
        out = torch.empty_like(x)
    check(load().rmsnorm(_p(x), _p(gamma), _p(out), M, H, float(eps), stream_handle(stream)))
    return out


def kv_append_rope(q, k, v, k_pool, v_pool, block_table, context_lens, theta, row_stride=0, err_flag=None,
                   n_q_heads=None, n_kv_heads=None, stream=None):
    """q [B][Hq][D] (rotated in place), k/v [B][Hkv][D]; pools [pages][Hkv][16][D]."""
    pages, Hkv, D, B = _paging(k_pool, v_pool, block_table, context_lens)
    _arg(err_flag, _I, "err_flag", optional=True)
    Hq = n_q_heads if n_q_heads is not None else q.shape[-2]
    if n_kv_heads is not None:
        Hkv = n_kv_heads
    check(load().kv_append_rope(_p(q), _p(k), _p(v), int(row_stride), _p(k_pool), _p(v_pool), pages,
                                _p(block_table), block_table.shape[1], _p(context_lens), B, Hq, Hkv, D,
                                float(theta), _p(err_flag), stream_handle(stream)))
    return q


def paged_gqa_decode_workspace_size(B, Hq, Hkv, max_context, partition_tokens=0, D=128):
    return int(load().paged_gqa_decode_workspace_size(B, Hq, Hkv, max_context, partition_tokens, D))


def paged_gqa_decode_default_partition(B, Hkv, max_context):
    return int(load().paged_gqa_decode_default_partition(B, Hkv, max_context))


def workspace_clear(ws, stream=None):
    check(load().w4a16_workspace_clear(_p(ws), ws.numel() * ws.element_size(), stream_handle(stream)))


def paged_gqa_decode(q, k_pool, v_pool, block_table, context_lens, max_context, sm_scale=None, partition_tokens=0,
                     workspace=None, out=None, err_flag=None, q_stride=0, n_q_heads=None, stream=None):
    """q [B][Hq][D] (or rows of pitch q_stride); returns out [B][Hq][D]."""
    pages, Hkv, D, B = _paging(k_pool, v_pool, block_table, context_lens)
    _arg(q, _H, "q")
    Hq = n_q_heads if n_q_heads is not None else q.shape[-2]
    if q.numel() < (B - 1) * (q_stride or Hq * D) + Hq * D:
        raise ValueError(f"q: {q.numel()} elements, too few for {B} rows of {Hq}x{D} at pitch {q_stride or Hq * D}")
    _arg(out, _H, "out", (B, Hq, D), optional=True)
    _arg(workspace, _U8, "workspace", optional=True)
    _arg(err_flag, _I, "err_flag", optional=True)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    lib = load()
    if workspace is None:
        nbytes = lib.paged_gqa_decode_workspace_size(B, Hq, Hkv, max_context, partition_tokens, D)
        workspace = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=k_pool.device)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float16, device=k_pool.device)
    check(lib.paged_gqa_decode(_p(q), int(q_stride), _p(k_pool), _p(v_pool), pages, _p(block_table),
                               block_table.shape[1], _p(context_lens), int(max_context), B, Hq, Hkv, D,
                               float(sm_scale), int(partition_tokens), _p(workspace),
                               workspace.numel() * workspace.element_size(), _p(out), _p(err_flag),
                               stream_handle(stream)))
    return out


def paged_gqa_decode_rope_append(qkv, k_pool, v_pool, block_table, context_lens, max_context, theta, n_q_heads,
                                 sm_scale=None, partition_tokens=0, workspace=None, out=None, err_flag=None,
                                 stream=None):
    """qkv rows [B][(Hq + 2 Hkv) D] (q | k_new | v_new); appends and attends."""
    pages, Hkv, D, B = _paging(k_pool, v_pool, block_table, context_lens)
    Hq = n_q_heads
    _arg(qkv, _H, "qkv", (B, None))
    if qkv.shape[1] < (Hq + 2 * Hkv) * D:
        raise ValueError(f"qkv: rows of {qkv.shape[1]}, need (Hq + 2 Hkv) D = {(Hq + 2 * Hkv) * D}")
    _arg(out, _H, "out", (B, Hq, D), optional=True)
    _arg(workspace, _U8, "workspace", optional=True)
    _arg(err_flag, _I, "err_flag", optional=True)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    lib = load()
    if workspace is None:
        nbytes = lib.paged_gqa_decode_workspace_size(B, Hq, Hkv, max_context, partition_tokens, D)
        workspace = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=k_pool.device)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float16, device=k_pool.device)
    check(lib.paged_gqa_decode_rope_append(_p(qkv), qkv.shape[-1] if qkv.dim() == 2 else 0, _p(k_pool), _p(v_pool),
                                           pages, _p(block_table), block_table.shape[1], _p(context_lens),
                                           int(max_context), B, Hq, Hkv, D, float(theta), float(sm_scale),
                                           int(partition_tokens), _p(workspace),
                                           workspace.numel() * workspace.element_size(), _p(out), _p(err_flag),
                                           stream_handle(stream)))
    return out


def _paging_fp8(k_pool, v_pool, k_scale, v_scale, block_table, context_lens):
    """(pages, Hkv, D, B) of FP8 pools: codes [pages][Hkv][16][D] uint8 and
    fp32 row scales [pages][Hkv][16]."""
    _arg(k_pool, _U8, "k_pool", (None, None, 16, None))
    pages, Hkv, _, D = k_pool.shape
    _arg(v_pool, _U8, "v_pool", tuple(k_pool.shape))
    _arg(k_scale, _F, "k_scale", (pages, Hkv, 16))
    _arg(v_scale, _F, "v_scale", (pages, Hkv, 16))
    _arg(block_table, _I, "block_table", (None, None))
    B = block_table.shape[0]
    _arg(context_lens, _I, "context_lens", (B,))
    return pages, Hkv, D, B


def kv_append_rope_fp8(q, k, v, k_pool, v_pool, k_scale, v_scale, block_table, context_lens, theta, row_stride=0,
                       err_flag=None, n_q_heads=None, n_kv_heads=None, stream=None):
    """kv_append_rope into FP8 pools: q [B][Hq][D] rotated in place; the
    rotated k row and the v row quantised (largest magnitude to 448) into
    their slot's codes and row scale."""
    pages, Hkv, D, B = _paging_fp8(k_pool, v_pool, k_scale, v_scale, block_table, context_lens)
    _arg(err_flag, _I, "err_flag", optional=True)
    Hq = n_q_heads if n_q_heads is not None else q.shape[-2]
    if n_kv_heads is not None:
        Hkv = n_kv_heads
    check(load().kv_append_rope_fp8(_p(q), _p(k), _p(v), int(row_stride), _p(k_pool), _p(v_pool), _p(k_scale),
                                    _p(v_scale), pages, _p(block_table), block_table.shape[1], _p(context_lens), B,
                                    Hq, Hkv, D, float(theta), _p(err_flag), stream_handle(stream)))
    return q


def paged_gqa_decode_fp8(q, k_pool, v_pool, k_scale, v_scale, block_table, context_lens, max_context, sm_scale=None,
                         partition_tokens=0, workspace=None, out=None, err_flag=None, qkv_theta=None,
                         n_q_heads=None, stream=None):
    """paged_gqa_decode over FP8 pools.  With qkv_theta given, q holds q|k|v
    rows (B, (Hq + 2 Hkv) D) and the call is the fused RoPE + FP8 append +
    attention (paged_gqa_decode_rope_append_fp8)."""
    pages, Hkv, D, B = _paging_fp8(k_pool, v_pool, k_scale, v_scale, block_table, context_lens)
    _arg(q, _H, "q")
    fuse = qkv_theta is not None
    Hq = n_q_heads if n_q_heads is not None else q.shape[-2]
    stride = q.shape[-1] if fuse else 0
    if fuse and (q.dim() != 2 or q.shape[0] != B or q.shape[1] < (Hq + 2 * Hkv) * D):
        raise ValueError(f"qkv: shape {tuple(q.shape)}, need ({B}, >= {(Hq + 2 * Hkv) * D})")
    if not fuse:
        _arg(q, _H, "q", (B, Hq, D))
    _arg(out, _H, "out", (B, Hq, D), optional=True)
    _arg(workspace, _U8, "workspace", optional=True)
    _arg(err_flag, _I, "err_flag", optional=True)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    lib = load()
    if workspace is None:
        nbytes = lib.paged_gqa_decode_workspace_size(B, Hq, Hkv, max_context, partition_tokens, D)
        workspace = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=k_pool.device)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float16, device=k_pool.device)
    common = (pages, _p(block_table), block_table.shape[1], _p(context_lens), int(max_context), B, Hq, Hkv, D)
    tail = (int(partition_tokens), _p(workspace), workspace.numel() * workspace.element_size(), _p(out),
            _p(err_flag), stream_handle(stream))
    if fuse:
        check(lib.paged_gqa_decode_rope_append_fp8(_p(q), int(stride), _p(k_pool), _p(v_pool), _p(k_scale),
                                                   _p(v_scale), *common, float(qkv_theta), float(sm_scale), *tail))
    else:
        check(lib.paged_gqa_decode_fp8(_p(q), 0, _p(k_pool), _p(v_pool), _p(k_scale), _p(v_scale), *common,
                                       float(sm_scale), *tail))
    return out


def embedding_gather(embed, tokens, out=None, err_flag=None, stream=None):
    _arg(embed, _H, "embed", (None, None))
    vocab, H = embed.shape
    _arg(tokens, _I, "tokens")
    B = tokens.numel()
    _arg(out, _H, "out", (B, H), optional=True)
    _arg(err_flag, _I, "err_flag", optional=True)
    if out is None:
        out = torch.empty((B, H), dtype=torch.float16, device=embed.device)
    check(load().embedding_gather(_p(embed), vocab, H, _p(tokens), B, _p(out), _p(err_flag),
                                  stream_handle(stream)))
    return out


def lm_head_argmax(x, lm_head, logits=None, tokens_out=None, workspace=None, want_logits=False, stream=None):
    B, H = _xk(x)
    _arg(lm_head, _H, "lm_head", (None, H))
    vocab = lm_head.shape[0]
    _arg(logits, _H, "logits", (B, vocab), optional=True)
    _arg(tokens_out, _I, "tokens_out", (B,), optional=True)
    _arg(workspace, _U8, "workspace", optional=True)
    lib = load()
    if workspace is None:
        workspace = torch.zeros(lib.lm_head_argmax_workspace_size(B, vocab), dtype=torch.uint8, device=x.device)
    if tokens_out is None:
        tokens_out = torch.empty(B, dtype=torch.int32, device=x.device)
    if logits is None and want_logits:
        logits = torch.empty((B, vocab), dtype=torch.float16, device=x.device)
    check(lib.lm_head_argmax(_p(x), B, H, _p(lm_head), vocab, _p(logits), _p(tokens_out), _p(workspace),
                             workspace.numel(), stream_handle(stream)))
    return tokens_out, logits


class Model:
    """Handle over w4a16_model_*: weights and pools stay owned by the caller
    (torch tensors kept alive here), the library owns its activation arena."""

    LAYER_KEYS = ("ln1", "ln2", "wq", "wk", "wv", "wo", "wg", "wu", "wd", "sq", "sk", "sv", "so", "sg", "su",
                  "sd", "bq", "bk", "bv", "k_pool", "v_pool", "k8", "v8", "k_scale", "v_scale")

    def __init__(self, cfg: dict, layers: list, embed=None, final_norm=None, lm_head=None, max_batch=1,
                 max_context=4096, num_pages=None, partition_tokens=0):
        self._lib = load()
        self.cfg = dict(cfg)
        self._keep = [embed, final_norm, lm_head]
        c = ModelConfig(cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["inter"],
                        len(layers), cfg.get("vocab", 0) if lm_head is not None else 0, float(cfg["eps"]),
                        float(cfg["theta"]), int(num_pages if num_pages is not None else
                                                 _layer_pool(layers[0]).shape[0]), int(partition_tokens))
        arr = (LayerWeights * max(1, len(layers)))()
        for i, lw in enumerate(layers):
            for key in self.LAYER_KEYS:
                t = lw.get(key)
                self._keep.append(t)
                setattr(arr[i], key, None if t is None else t.data_ptr())
        self._layers_arr = arr
        w = ModelWeights(_p(embed), _p(final_norm), _p(lm_head),
                         ctypes.cast(arr, ctypes.POINTER(LayerWeights)))
        h = ctypes.c_void_p()
        check(self._lib.w4a16_model_create(ctypes.byref(c), ctypes.byref(w), int(max_batch), int(max_context),
                                           ctypes.byref(h)))
        self._h = h
        self.max_batch, self.max_context = max_batch, max_context

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.w4a16_model_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def err_flag_ptr(self) -> int:
        return int(self._lib.w4a16_model_err_flag(self._h) or 0)

    def hidden(self, B=1, out=None, stream=None):
        """Final hidden states (pre final-norm) of the last decode step."""
        if out is None:
            out = torch.empty((B, self.cfg["hidden"]), dtype=torch.float16, device="cuda")
        check(self._lib.w4a16_model_hidden(self._h, _p(out), int(B), stream_handle(stream)))
        return out

    ACTIVATIONS = {"hidden": (0, "hidden"), "qkv": (1, None), "attn": (2, None), "resid": (3, "hidden"),
                   "mlp": (4, "inter")}

    def activation(self, name, B=1, stream=None):
        """Copy of an arena activation buffer left by the last layer or step:
        hidden, qkv, attn, resid (x + o) or mlp (silu(gate) * up)."""
        which, key = self.ACTIVATIONS[name]
        c = self.cfg
        width = {"qkv": (c["n_q_heads"] + 2 * c["n_kv_heads"]) * c["head_dim"],
                 "attn": c["n_q_heads"] * c["head_dim"]}.get(name) or c[key]
        out = torch.empty((B, width), dtype=torch.float16, device="cuda")
        check(self._lib.w4a16_model_activation(self._h, which, _p(out), int(B), stream_handle(stream)))
        return out

    def check_errors(self, stream=None) -> int:
        """Status code of the device error word (blocks; clears the word)."""
        return int(self._lib.w4a16_model_check_errors(self._h, stream_handle(stream)))

    def _paging_args(self, B, block_table, context_lens):
        _arg(block_table, _I, "block_table", (B, None))
        _arg(context_lens, _I, "context_lens", (B,))

    def layer(self, i, x, block_table, context_lens, stream=None):
        _arg(x, _H, "x", (None, self.cfg["hidden"]))
        self._paging_args(x.shape[0], block_table, context_lens)
        check(self._lib.w4a16_model_layer(self._h, int(i), _p(x), _p(block_table), block_table.shape[1],
                                          _p(context_lens), x.shape[0], stream_handle(stream)))
        return x

    def decode_step(self, tokens_in, tokens_out, block_table, context_lens, logits=None, use_graph=True,
                    stream=None):
        _arg(tokens_in, _I, "tokens_in")
        B = tokens_in.numel()
        _arg(tokens_out, _I, "tokens_out", tuple(tokens_in.shape))
        self._paging_args(B, block_table, context_lens)
        _arg(logits, _H, "logits", (B, self.cfg.get("vocab", 0)), optional=True)
        check(self._lib.decode_step(self._h, _p(tokens_in), _p(tokens_out), _p(block_table), block_table.shape[1],
                                    _p(context_lens), tokens_in.numel(), _p(logits), int(bool(use_graph)),
                                    stream_handle(stream)))
        return tokens_out

    def kernel_count(self, B=1) -> int:
        return int(self._lib.decode_step_kernel_count(self._h, int(B)))

    def prefill(self, tokens, block_table, context_lens, token_out=None, logits=None, workspace=None, stream=None):
        """One sequence's prompt tokens [T] in one pass: writes their KV pages,
        advances context_lens[0] by T, returns the greedy next token [1]."""
        _arg(tokens, _I, "tokens")
        T = tokens.numel()
        _arg(block_table, _I, "block_table", (1, None))
        _arg(context_lens, _I, "context_lens", (1,))
        _arg(logits, _H, "logits", (1, self.cfg.get("vocab", 0)), optional=True)
        lib = self._lib
        need = int(lib.w4a16_prefill_workspace_size(self._h, T, block_table.shape[1]))
        if workspace is None:
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=tokens.device)
        _arg(workspace, _U8, "workspace")
        if token_out is None:
            token_out = torch.empty(1, dtype=torch.int32, device=tokens.device)
        _arg(token_out, _I, "token_out", (1,))
        check(lib.w4a16_prefill(self._h, _p(tokens), T, _p(block_table), block_table.shape[1], _p(context_lens),
                                _p(token_out), _p(logits), _p(workspace), workspace.numel(), stream_handle(stream)))
        return token_out

    PATHS = {"auto": 0, "kernels": 1, "persistent": 2}

    def set_decode_path(self, path: str) -> None:
        """'auto' (persistent kernel where it applies), 'kernels' or
        'persistent' (raises if the model is outside what it covers)."""
        check(self._lib.w4a16_model_set_decode_path(self._h, self.PATHS[path]))

    def decode_path(self, B=1) -> str:
        """The path decode_step takes for B sequences."""
        code = int(self._lib.w4a16_model_decode_path(self._h, int(B)))
        return {1: "kernels", 2: "persistent"}[code]


class Batcher:
    """Continuous batching over a Model (w4a16_batcher_*): sequences are
    queued with submit(), step() runs one decode step over the active ones
    (admitting queued sequences as others finish, pages handed out and
    reclaimed by the library's allocator), poll() reads a sequence's tokens."""

    def __init__(self, model: "Model", num_pages: int, max_batch: int, max_blocks: int, max_context: int):
        self._lib = load()
        self.model = model
        h = ctypes.c_void_p()
        check(self._lib.w4a16_batcher_create(model._h, int(num_pages), int(max_batch), int(max_blocks),
                                             int(max_context), ctypes.byref(h)))
        self._h = h

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.w4a16_batcher_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def submit(self, prompt, max_new_tokens: int) -> int:
        import numpy as np
        p = np.ascontiguousarray(prompt, dtype=np.int32)
        sid = ctypes.c_int()
        check(self._lib.w4a16_batcher_submit(self._h, p.ctypes.data, int(p.size), int(max_new_tokens),
                                             ctypes.byref(sid)))
        return sid.value

    def step(self, stream=None) -> int:
        n = ctypes.c_int()
        check(self._lib.w4a16_batcher_step(self._h, stream_handle(stream), ctypes.byref(n)))
        return n.value

    def poll(self, seq_id: int):
        """(generated tokens so far, finished?)"""
        import numpy as np
        n, done = ctypes.c_int(), ctypes.c_int()
        check(self._lib.w4a16_batcher_poll(self._h, int(seq_id), None, 0, ctypes.byref(n), ctypes.byref(done)))
        out = np.zeros(max(1, n.value), np.int32)
        check(self._lib.w4a16_batcher_poll(self._h, int(seq_id), out.ctypes.data, n.value, ctypes.byref(n),
                                           ctypes.byref(done)))
        return out[:n.value], bool(done.value)

    def stats(self) -> dict:
        st, pre = ctypes.c_long(), ctypes.c_long()
        wt, ac, fp = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        check(self._lib.w4a16_batcher_stats(self._h, ctypes.byref(st), ctypes.byref(pre), ctypes.byref(wt),
                                            ctypes.byref(ac), ctypes.byref(fp)))
        return {"steps": st.value, "preemptions": pre.value, "waiting": wt.value, "active": ac.value,
                "free_pages": fp.value}


def device_pool(case: dict, layer: int, which: str, device="cuda"):
    """One layer's K or V pool of a ``synth.model_case`` on the device: zeros,
    with the pages the block tables name filled in."""
    cfg = case["cfg"]
    p = torch.zeros((case["pool_pages"], cfg["n_kv_heads"], 16, cfg["head_dim"]), dtype=torch.float16,
                    device=device)
    idx = torch.from_numpy(case["used_pages"]).to(device)
    p[idx] = torch.from_numpy(case[which + "_used"][layer]).to(device)
    return p


def _layer_pool(layer: dict):
    return layer["k_pool"] if layer.get("k_pool") is not None else layer["k8"]


def device_layer(w: dict, k_pool, v_pool, device="cuda") -> dict:
    """Move one layer's numpy weights (as drawn by ``synth``) and its pools to
    the device as torch tensors (uint32 words travel as int32).  A pool given
    as a (codes uint8, scales fp32) pair makes the layer's KV cache FP8
    (E4M3) pages."""
    import numpy as np

    out = {}
    for key, a in w.items():
        if a is None:
            out[key] = None
            continue
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint32:
            a = a.view(np.int32)
        out[key] = torch.from_numpy(a).to(device)
    dev = lambda a: a if isinstance(a, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(a)).to(device)
    if isinstance(k_pool, tuple):
        (k8, ks), (v8, vs) = k_pool, v_pool
        out["k_pool"] = out["v_pool"] = None
        out["k8"], out["k_scale"], out["v8"], out["v_scale"] = dev(k8), dev(ks), dev(v8), dev(vs)
        for key, dt in (("k8", torch.uint8), ("v8", torch.uint8), ("k_scale", torch.float32),
                        ("v_scale", torch.float32)):
            if out[key].dtype != dt or not out[key].is_contiguous():
                raise ValueError(f"{key}: {dt} contiguous expected")
        return out
    for key, a in (("k_pool", k_pool), ("v_pool", v_pool)):
        out[key] = dev(a)
    return out
