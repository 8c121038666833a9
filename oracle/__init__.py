"""CPU oracle for the W4A16 + paged-GQA decode path (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The product library never does.

The arithmetic lives in ``oracle.c`` (plain C, fp64).  This module compiles it
with gcc on first use and exposes numpy-friendly wrappers; it holds no method
arithmetic of its own beyond reshaping arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


class Config(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int), ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int), ("inter", ctypes.c_int), ("n_layers", ctypes.c_int),
        ("vocab", ctypes.c_int), ("eps", ctypes.c_double), ("theta", ctypes.c_double),
    ]


_P = ctypes.c_void_p


class Layer(ctypes.Structure):
    _fields_ = [(n, _P) for n in (
        "ln1", "ln2", "wq", "wk", "wv", "wo", "wg", "wu", "wd",
        "sq", "sk", "sv", "so", "sg", "su", "sd", "bq", "bk", "bv", "k_pool", "v_pool",
        "k8", "v8", "k_scale", "v_scale")]


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            l = ctypes.CDLL(build())
            i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            sig = {
                "orc_half_to_double": (dbl, [ctypes.c_uint16]),
                "orc_double_to_half": (ctypes.c_uint16, [dbl]),
                "orc_half_to_double_array": (None, [_P, i64, _P]),
                "orc_double_to_half_array": (None, [_P, i64, _P]),
                "orc_num_threads": (i32, []),
                "orc_set_num_threads": (None, [i32]),
                "orc_unpack_code": (i32, [ctypes.c_uint32, i32]),
                "orc_pack_int4": (None, [_P, i64, i64, _P]),
                "orc_unpack_int4": (None, [_P, i64, i64, _P]),
                "orc_dequant": (None, [_P, _P, i64, i64, _P]),
                "orc_quantize": (None, [_P, i64, i64, _P, _P]),
                "orc_w4a16_gemv": (None, [_P, i32, i32, _P, _P, i32, _P, _P, _P]),
                "orc_fp16_gemv": (None, [_P, i32, _P, i32, _P]),
                "orc_argmax": (i64, [_P, i64]),
                "orc_rmsnorm": (None, [_P, _P, i32, i32, dbl, _P]),
                "orc_rope_inv_freq": (ctypes.c_float, [i32, i32, dbl]),
                "orc_rope_angle": (ctypes.c_float, [i32, i32, i32, dbl]),
                "orc_rope": (None, [_P, i32, i32, i32, dbl]),
                "orc_kv_append": (None, [_P, _P, _P, _P, _P, i32, _P, i32, i32, i32]),
                "orc_gather_kv": (None, [_P, _P, i32, i32, i32, _P]),
                "orc_attention": (None, [_P, _P, _P, i32, i32, i32, i32, dbl, _P]),
                "orc_attention_probs": (None, [_P, _P, i32, i32, i32, i32, dbl, i32, _P]),
                "orc_paged_attention": (None, [_P, _P, _P, _P, i32, _P, i32, i32, i32, i32, dbl, _P]),
                "orc_attention_split_combine": (None, [_P, _P, _P, i32, i32, i32, i32, dbl, i32, i32, _P]),
                "orc_silu_mul": (None, [_P, _P, i64, _P]),
                "orc_e4m3_to_double": (dbl, [ctypes.c_uint8]),
                "orc_float_to_e4m3": (ctypes.c_uint8, [ctypes.c_float]),
                "orc_fp8_quantize_row": (None, [_P, i32, _P, _P]),
                "orc_kv_append_fp8": (None, [_P, _P, _P, _P, _P, _P, _P, i32, _P, i32, i32, i32]),
                "orc_paged_attention_fp8": (None, [_P, _P, _P, _P, _P, _P, i32, _P, i32, i32, i32, i32, dbl,
                                                   _P]),
                "orc_decoder_layer": (None, [ctypes.POINTER(Config), ctypes.POINTER(Layer), _P, _P, i32, _P, i32]),
                "orc_decode_step": (None, [ctypes.POINTER(Config), ctypes.POINTER(Layer), i32, _P, _P, _P,
                                           _P, _P, i32, _P, i32, _P, _P, _P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(l, name)
                fn.restype = res
                fn.argtypes = args
            _lib = l
    return _lib


# ---------------------------------------------------------------------------
# numpy wrappers.  fp16 arrays travel as float16 (bit-identical to uint16).
# ---------------------------------------------------------------------------

def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data


def num_threads() -> int:
    return lib().orc_num_threads()


def set_num_threads(n: int) -> None:
    """Threads the oracle's parallel loops use from now on (for timing it on
    one core and on all host cores)."""
    lib().orc_set_num_threads(int(n))


def half_to_double(h: np.ndarray) -> np.ndarray:
    h = _c(h, np.float16)
    out = np.empty(h.shape, np.float64)
    lib().orc_half_to_double_array(_ptr(h), h.size, _ptr(out))
    return out


def double_to_half(d: np.ndarray) -> np.ndarray:
    d = _c(d, np.float64)
    out = np.empty(d.shape, np.float16)
    lib().orc_double_to_half_array(_ptr(d), d.size, _ptr(out))
    return out


def unpack_code(word: int, i: int) -> int:
    return lib().orc_unpack_code(word, i)


def pack_int4(q: np.ndarray) -> np.ndarray:
    q = _c(q, np.int8)
    N, K = q.shape
    out = np.empty((N, K // 8), np.uint32)
    lib().orc_pack_int4(_ptr(q), N, K, _ptr(out))
    return out


def unpack_int4(qw: np.ndarray, K: int) -> np.ndarray:
    qw = _c(qw, np.uint32)
    N = qw.shape[0]
    out = np.empty((N, K), np.int8)
    lib().orc_unpack_int4(_ptr(qw), N, K, _ptr(out))
    return out


def dequant(qw: np.ndarray, scales: np.ndarray, K: int) -> np.ndarray:
    qw, scales = _c(qw, np.uint32), _c(scales, np.float16)
    N = qw.shape[0]
    out = np.empty((N, K), np.float64)
    lib().orc_dequant(_ptr(qw), _ptr(scales), N, K, _ptr(out))
    return out


def quantize(w: np.ndarray):
    w = _c(w, np.float64)
    N, K = w.shape
    qw = np.empty((N, K // 8), np.uint32)
    s = np.empty((N, K // 128), np.float16)
    lib().orc_quantize(_ptr(w), N, K, _ptr(qw), _ptr(s))
    return qw, s


def w4a16_gemv(x, qw, scales, bias=None, residual=None):
    x = _c(np.atleast_2d(x), np.float16)
    qw, scales = _c(qw, np.uint32), _c(scales, np.float16)
    M, K = x.shape
    N = qw.shape[0]
    bias = None if bias is None else _c(bias, np.float16)
    residual = None if residual is None else _c(residual, np.float16).reshape(M, N)
    y = np.empty((M, N), np.float16)
    lib().orc_w4a16_gemv(_ptr(x), M, K, _ptr(qw), _ptr(scales), N, _ptr(bias), _ptr(residual), _ptr(y))
    return y


def fp16_gemv(x, w):
    x, w = _c(x, np.float16).reshape(-1), _c(w, np.float16)
    N, K = w.shape
    out = np.empty(N, np.float64)
    lib().orc_fp16_gemv(_ptr(x), K, _ptr(w), N, _ptr(out))
    return out


def argmax(v) -> int:
    v = _c(v, np.float64)
    return int(lib().orc_argmax(_ptr(v), v.size))


def rmsnorm(x, gamma, eps):
    x = _c(np.atleast_2d(x), np.float16)
    gamma = _c(gamma, np.float16)
    M, H = x.shape
    y = np.empty_like(x)
    lib().orc_rmsnorm(_ptr(x), _ptr(gamma), M, H, eps, _ptr(y))
    return y


def rope_inv_freq(i: int, D: int, theta: float) -> float:
    return lib().orc_rope_inv_freq(i, D, theta)


def rope_angle(pos: int, i: int, D: int, theta: float) -> float:
    return lib().orc_rope_angle(pos, i, D, theta)


def rope(x, pos: int, theta: float):
    """x [nheads][D] fp16 -> rotated copy."""
    x = np.array(x, dtype=np.float16, order="C", copy=True)
    nheads, D = x.reshape(-1, x.shape[-1]).shape
    lib().orc_rope(_ptr(x), nheads, D, pos, theta)
    return x


def kv_append(k, v, k_pool, v_pool, block_table, context_lens):
    """In place on k_pool / v_pool.  k, v [B][Hkv][D]."""
    k, v = _c(k, np.float16), _c(v, np.float16)
    block_table, context_lens = _c(block_table, np.int32), _c(context_lens, np.int32)
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    B, Hkv, D = k.shape
    lib().orc_kv_append(_ptr(k), _ptr(v), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                        block_table.shape[1], _ptr(context_lens), B, Hkv, D)


def gather_kv(pool, block_table_row, L: int):
    pool = _c(pool, np.float16)
    row = _c(block_table_row, np.int32)
    _, Hkv, _, D = pool.shape
    out = np.empty((L, Hkv, D), np.float16)
    lib().orc_gather_kv(_ptr(pool), _ptr(row), L, Hkv, D, _ptr(out))
    return out


def attention(q, k, v, scale):
    """q [Hq][D], k/v [L][Hkv][D] -> [Hq][D] fp16."""
    q, k, v = _c(q, np.float16), _c(k, np.float16), _c(v, np.float16)
    Hq, D = q.shape
    L, Hkv, _ = k.shape
    out = np.empty((Hq, D), np.float16)
    lib().orc_attention(_ptr(q), _ptr(k), _ptr(v), Hq, Hkv, D, L, scale, _ptr(out))
    return out


def attention_probs(q, k, scale, h: int):
    q, k = _c(q, np.float16), _c(k, np.float16)
    Hq, D = q.shape
    L, Hkv, _ = k.shape
    p = np.empty(L, np.float64)
    lib().orc_attention_probs(_ptr(q), _ptr(k), Hq, Hkv, D, L, scale, h, _ptr(p))
    return p


def paged_attention(q, k_pool, v_pool, block_table, context_lens, scale):
    q = _c(q, np.float16)
    k_pool, v_pool = _c(k_pool, np.float16), _c(v_pool, np.float16)
    block_table, context_lens = _c(block_table, np.int32), _c(context_lens, np.int32)
    B, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    out = np.empty((B, Hq, D), np.float16)
    lib().orc_paged_attention(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                              block_table.shape[1], _ptr(context_lens), B, Hq, Hkv, D, scale, _ptr(out))
    return out


def attention_split_combine(q, k, v, scale, h: int, part: int):
    q, k, v = _c(q, np.float16), _c(k, np.float16), _c(v, np.float16)
    Hq, D = q.shape
    L, Hkv, _ = k.shape
    out = np.empty(D, np.float64)
    lib().orc_attention_split_combine(_ptr(q), _ptr(k), _ptr(v), Hq, Hkv, D, L, scale, h, part, _ptr(out))
    return out


def e4m3_to_double(code: int) -> float:
    """Value of one FP8 E4M3 code (NaN for S.1111.111)."""
    return lib().orc_e4m3_to_double(int(code) & 0xFF)


def float_to_e4m3(f: float) -> int:
    """E4M3 code of an fp32 value: round to nearest even, saturating at 448."""
    return int(lib().orc_float_to_e4m3(float(f)))


def fp8_quantize_row(x):
    """(codes uint8 [D], fp32 scale) of one fp16 row: the row's largest
    magnitude maps to 448."""
    x = _c(x, np.float16).ravel()
    codes = np.empty(x.size, np.uint8)
    sc = np.zeros(1, np.float32)
    lib().orc_fp8_quantize_row(_ptr(x), x.size, _ptr(codes), _ptr(sc))
    return codes, float(sc[0])


def kv_append_fp8(k, v, k_pool, v_pool, k_scale, v_scale, block_table, context_lens):
    """In place: quantise k[b], v[b] ([B][Hkv][D] fp16, k already rotated)
    into slot context_lens[b]-1 of the FP8 pools ([pages][Hkv][16][D] uint8)
    and their fp32 row scales ([pages][Hkv][16])."""
    k, v = _c(k, np.float16), _c(v, np.float16)
    for a, dt in ((k_pool, np.uint8), (v_pool, np.uint8), (k_scale, np.float32), (v_scale, np.float32)):
        assert a.dtype == dt and a.flags.c_contiguous
    block_table, context_lens = _c(block_table, np.int32), _c(context_lens, np.int32)
    B, Hkv, D = k.shape
    lib().orc_kv_append_fp8(_ptr(k), _ptr(v), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale),
                            _ptr(block_table), block_table.shape[1], _ptr(context_lens), B, Hkv, D)


def paged_attention_fp8(q, k_pool, v_pool, k_scale, v_scale, block_table, context_lens, scale):
    q = _c(q, np.float16)
    k_pool, v_pool = _c(k_pool, np.uint8), _c(v_pool, np.uint8)
    k_scale, v_scale = _c(k_scale, np.float32), _c(v_scale, np.float32)
    block_table, context_lens = _c(block_table, np.int32), _c(context_lens, np.int32)
    B, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    out = np.empty((B, Hq, D), np.float16)
    lib().orc_paged_attention_fp8(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale),
                                  _ptr(block_table), block_table.shape[1], _ptr(context_lens), B, Hq, Hkv, D,
                                  scale, _ptr(out))
    return out


def silu_mul(g, u):
    g, u = _c(g, np.float16), _c(u, np.float16)
    m = np.empty_like(g)
    lib().orc_silu_mul(_ptr(g), _ptr(u), g.size, _ptr(m))
    return m


# ---------------------------------------------------------------------------
# Whole layer / whole model.  Weights are dicts of numpy arrays named as in
# the synthetic-input module (ln1, ln2, wq..wd, sq..sd, bq/bk/bv optional).
# ---------------------------------------------------------------------------

def make_config(cfg: dict) -> Config:
    return Config(cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["inter"],
                  cfg["n_layers"], cfg.get("vocab", 0), cfg["eps"], cfg["theta"])


def make_layer(w: dict, k_pool, v_pool, keep: list) -> Layer:
    """k_pool / v_pool: fp16 pools, or FP8 pools as (codes uint8, scales fp32)
    pairs (updated in place by the layer's append)."""
    lay = Layer()
    for name in ("ln1", "ln2", "sq", "sk", "sv", "so", "sg", "su", "sd"):
        a = _c(w[name], np.float16)
        keep.append(a)
        setattr(lay, name, a.ctypes.data)
    for name in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"):
        a = _c(w[name], np.uint32)
        keep.append(a)
        setattr(lay, name, a.ctypes.data)
    for name in ("bq", "bk", "bv"):
        if w.get(name) is not None:
            a = _c(w[name], np.float16)
            keep.append(a)
            setattr(lay, name, a.ctypes.data)
    if isinstance(k_pool, tuple):
        (k8, ks), (v8, vs) = k_pool, v_pool
        for a, dt in ((k8, np.uint8), (v8, np.uint8), (ks, np.float32), (vs, np.float32)):
            assert a.dtype == dt and a.flags.c_contiguous
        lay.k8, lay.v8, lay.k_scale, lay.v_scale = k8.ctypes.data, v8.ctypes.data, ks.ctypes.data, vs.ctypes.data
        return lay
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    assert k_pool.dtype == np.float16 and v_pool.dtype == np.float16
    lay.k_pool = k_pool.ctypes.data
    lay.v_pool = v_pool.ctypes.data
    return lay


def decoder_layer(cfg: dict, w: dict, x, k_pool, v_pool, block_table, context_lens):
    """Returns the layer output; appends into k_pool / v_pool in place."""
    keep: list = []
    c = make_config(cfg)
    lay = make_layer(w, k_pool, v_pool, keep)
    x = np.array(np.atleast_2d(x), dtype=np.float16, order="C", copy=True)
    block_table, context_lens = _c(block_table, np.int32), _c(context_lens, np.int32)
    lib().orc_decoder_layer(ctypes.byref(c), ctypes.byref(lay), _ptr(x), _ptr(block_table),
                            block_table.shape[1], _ptr(context_lens), x.shape[0])
    return x


def decode_step(cfg: dict, layers: list, k_pools: list, v_pools: list, embed, final_norm, lm_head,
                tokens_in, block_table, context_lens, n_layers_run=None, want_logits=False):
    """Returns (tokens_out [B], logits fp16 [B][V] or None, final hidden [B][H])."""
    keep: list = []
    c = make_config(cfg)
    n_run = len(layers) if n_layers_run is None else n_layers_run
    arr = (Layer * max(1, len(layers)))()
    for i, w in enumerate(layers):
        arr[i] = make_layer(w, k_pools[i], v_pools[i], keep)
    embed, final_norm, lm_head = _c(embed, np.float16), _c(final_norm, np.float16), _c(lm_head, np.float16)
    tokens_in = _c(tokens_in, np.int32)
    block_table, context_lens = _c(block_table, np.int32), _c(context_lens, np.int32)
    B = tokens_in.size
    tokens_out = np.empty(B, np.int32)
    logits = np.empty((B, cfg["vocab"]), np.float16) if want_logits else None
    hidden = np.empty((B, cfg["hidden"]), np.float16)
    lib().orc_decode_step(ctypes.byref(c), arr, n_run, _ptr(embed), _ptr(final_norm), _ptr(lm_head),
                          _ptr(tokens_in), _ptr(block_table), block_table.shape[1], _ptr(context_lens),
                          B, _ptr(tokens_out), _ptr(logits), _ptr(hidden))
    return tokens_out, logits, hidden
