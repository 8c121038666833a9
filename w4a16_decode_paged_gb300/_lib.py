"""ctypes binding of libw4a16_gb300.so (include/w4a16.h).

Argument marshalling only: tensors are passed as device pointers, sizes as
ints, and the current torch CUDA stream as the cudaStream_t.  Every step of
the decode path runs in the library's kernels; if the library is missing the
calls raise instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I32 = ctypes.c_int
F32 = ctypes.c_float
SZ = ctypes.c_size_t

ERR_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "ALIGNMENT", 3: "SHAPE", 4: "CUDA", 5: "CAPTURE",
             6: "DEVICE_BOUNDS", 7: "TIMEOUT", 8: "NO_PAGES"}


class W4A16Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERR_NAMES.get(code, code)}: {msg}")
        self.code = code


class ModelConfig(ctypes.Structure):
    _fields_ = [("hidden", I32), ("n_q_heads", I32), ("n_kv_heads", I32), ("head_dim", I32), ("inter", I32),
                ("n_layers", I32), ("vocab", I32), ("eps", F32), ("theta", F32), ("num_pages", I32),
                ("partition_tokens", I32)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, P) for n in ("ln1", "ln2", "wq", "wk", "wv", "wo", "wg", "wu", "wd", "sq", "sk", "sv", "so",
                                 "sg", "su", "sd", "bq", "bk", "bv", "k_pool", "v_pool",
                                 "k8", "v8", "k_scale", "v_scale")]


class ModelWeights(ctypes.Structure):
    _fields_ = [("embed", P), ("final_norm", P), ("lm_head", P), ("layers", ctypes.POINTER(LayerWeights))]


# name -> (restype, argtypes); mirrors include/w4a16.h
SIGNATURES = {
    "w4a16_last_error": (ctypes.c_char_p, []),
    "w4a16_version": (I32, []),
    "w4a16_gemv": (I32, [P, I32, I32, P, P, I32, P, P, P, P]),
    "w4a16_gemm": (I32, [P, I32, I32, P, P, I32, P, P, P, P, SZ, P]),
    "w4a16_gemm_silu_mul": (I32, [P, I32, I32, P, P, P, P, I32, P, P, SZ, P]),
    "w4a16_gemm_workspace_size": (SZ, [I32, I32, I32, I32]),
    "w4a16_debug_set_wait_limit_ns": (ctypes.c_ulonglong, [ctypes.c_ulonglong]),
    "lm_head_logits_batched": (I32, [P, I32, I32, P, I32, P, P]),
    "argmax_rows": (I32, [P, I32, I32, P, P, P]),
    "w4a16_gemv_rmsnorm": (I32, [P, P, F32, I32, I32, P, P, I32, P, P, P]),
    "w4a16_gemv_silu_mul": (I32, [P, P, F32, I32, I32, P, P, P, P, I32, P, P]),
    "rmsnorm": (I32, [P, P, P, I32, I32, F32, P]),
    "kv_append_rope": (I32, [P, P, P, I32, P, P, I32, P, I32, P, I32, I32, I32, I32, F32, P, P]),
    "paged_gqa_decode": (I32, [P, I32, P, P, I32, P, I32, P, I32, I32, I32, I32, I32, F32, I32, P, SZ, P, P, P]),
    "paged_gqa_decode_rope_append": (I32, [P, I32, P, P, I32, P, I32, P, I32, I32, I32, I32, I32, F32, F32, I32, P,
                                           SZ, P, P, P]),
    "paged_gqa_decode_noalloc": (I32, [P, I32, P, P, I32, P, I32, P, I32, I32, I32, I32, I32, F32, I32, P, P, P]),
    "paged_gqa_decode_fp8": (I32, [P, I32, P, P, P, P, I32, P, I32, P, I32, I32, I32, I32, I32, F32, I32, P, SZ, P,
                                   P, P]),
    "paged_gqa_decode_rope_append_fp8": (I32, [P, I32, P, P, P, P, I32, P, I32, P, I32, I32, I32, I32, I32, F32, F32,
                                               I32, P, SZ, P, P, P]),
    "kv_append_rope_fp8": (I32, [P, P, P, I32, P, P, P, P, I32, P, I32, P, I32, I32, I32, I32, F32, P, P]),
    "paged_gqa_decode_workspace_size": (SZ, [I32, I32, I32, I32, I32, I32]),
    "paged_gqa_decode_default_partition": (I32, [I32, I32, I32]),
    "w4a16_workspace_clear": (I32, [P, SZ, P]),
    "embedding_gather": (I32, [P, I32, I32, P, I32, P, P, P]),
    "lm_head_argmax": (I32, [P, I32, I32, P, I32, P, P, P, SZ, P]),
    "lm_head_argmax_workspace_size": (SZ, [I32, I32]),
    "w4a16_model_create": (I32, [ctypes.POINTER(ModelConfig), ctypes.POINTER(ModelWeights), I32, I32,
                                 ctypes.POINTER(P)]),
    "w4a16_model_destroy": (None, [P]),
    "w4a16_model_err_flag": (P, [P]),
    "w4a16_model_check_errors": (I32, [P, P]),
    "w4a16_model_hidden": (I32, [P, P, I32, P]),
    "w4a16_model_activation": (I32, [P, I32, P, I32, P]),
    "w4a16_model_layer": (I32, [P, I32, P, P, I32, P, I32, P]),
    "decode_step": (I32, [P, P, P, P, I32, P, I32, P, I32, P]),
    "decode_step_kernel_count": (I32, [P, I32]),
    "w4a16_model_set_decode_path": (I32, [P, I32]),
    "w4a16_prefill_workspace_size": (SZ, [P, I32, I32]),
    "w4a16_prefill": (I32, [P, P, I32, P, I32, P, P, P, P, SZ, P]),
    "w4a16_page_allocator_create": (I32, [I32, ctypes.POINTER(P)]),
    "w4a16_page_allocator_destroy": (None, [P]),
    "w4a16_page_alloc": (I32, [P, I32, P]),
    "w4a16_page_free": (I32, [P, P, I32]),
    "w4a16_page_free_count": (I32, [P]),
    "w4a16_seq_reserve": (I32, [P, P, I32, I32]),
    "w4a16_seq_release": (I32, [P, P, I32]),
    "w4a16_batcher_create": (I32, [P, I32, I32, I32, I32, ctypes.POINTER(P)]),
    "w4a16_batcher_destroy": (None, [P]),
    "w4a16_batcher_submit": (I32, [P, P, I32, I32, ctypes.POINTER(I32)]),
    "w4a16_batcher_step": (I32, [P, P, ctypes.POINTER(I32)]),
    "w4a16_batcher_poll": (I32, [P, I32, P, I32, ctypes.POINTER(I32), ctypes.POINTER(I32)]),
    "w4a16_batcher_stats": (I32, [P, ctypes.POINTER(ctypes.c_long), ctypes.POINTER(ctypes.c_long),
                                  ctypes.POINTER(I32), ctypes.POINTER(I32), ctypes.POINTER(I32)]),
    "w4a16_model_decode_path": (I32, [P, I32]),
}


def lib_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load the built library; raises if it has not been built.  Setting
    W4A16_TRACE=1 loads the kernel-timeline build instead."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.TRACE_LIB if os.environ.get("W4A16_TRACE") == "1" else _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            if hasattr(lib, "w4a16_trace_start"):
                lib.w4a16_trace_start.restype = I32
                lib.w4a16_trace_start.argtypes = [P, ctypes.c_uint]
                lib.w4a16_trace_count.restype = ctypes.c_uint
                lib.w4a16_trace_count.argtypes = []
            _lib = lib
    return _lib


def check(rc: int) -> None:
    if rc != 0:
        msg = load().w4a16_last_error()
        raise W4A16Error(rc, msg.decode() if msg else "")
