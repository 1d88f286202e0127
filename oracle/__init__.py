"""CPU oracle for MFA decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its cpu_baseline
leg and its reference arm) may import this package.  The product path
(``decode_attention_02_gb300``) never imports it and shares no code with it.

``mfa_oracle.c`` is the plain fp64 definition of softmax(q K^T * scale) V over
the paged cache (Step-3, paperlayer.ai/abs/2507.19427v1, sections 2 and 5), for
MFA's one shared key/value head and for the grouped-head (GQA-style) and
shared-latent (MLA-style) caches of the attention designs the page compares;
this module compiles it with gcc and calls it through ctypes.

Pins (tests/test_oracle.py): torch SDPA in float64 on a dense gather done by
numpy indexing, scipy logsumexp for lse, the two-token logistic closed form,
L=1 -> v_0, constant K -> mean of V, key-shift and block-permutation
invariance, convex hull, split/merge identity, and every e4m3 code against
torch.float8_e4m3fn.  The KV append (tests/test_oracle_append.py): the e4m3
encoder against torch.float8_e4m3fn on every fp32 value it can decide
differently (codes, midpoints, their neighbours), round trips of every code,
saturation, signed zeros; the append against the dequantisation error bound,
the row maximum landing on code 448, and untouched slots left unchanged.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mfa_oracle.c")
_LIB = os.path.join(_HERE, "libmfa_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags: same results on x86_64 and aarch64)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def load_library(path: str):
    """Load a compiled oracle library and declare its signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.mfa_oracle_decode.argtypes = [I, I, I, I, I, I, I, P, P, P, P, P, P, P, P, P,
                                      ctypes.c_double, P, P, I]
    lib.mfa_oracle_decode.restype = I
    lib.mfa_oracle_combine.argtypes = [I, ctypes.c_long, I, P, P, P, P]
    lib.mfa_oracle_combine.restype = I
    lib.mfa_oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.mfa_oracle_e4m3_to_double.restype = ctypes.c_double
    lib.mfa_oracle_num_cpus.argtypes = []
    lib.mfa_oracle_num_cpus.restype = I
    lib.mfa_oracle_e4m3_from_float.argtypes = [ctypes.c_float]
    lib.mfa_oracle_e4m3_from_float.restype = ctypes.c_uint8
    lib.mfa_oracle_e4m3_from_float_array.argtypes = [P, ctypes.c_long, P]
    lib.mfa_oracle_e4m3_from_float_array.restype = None
    lib.mfa_oracle_kv_append.argtypes = [I, I, I, I, I, I, I, P, P, P, P, P, P, P, P]
    lib.mfa_oracle_kv_append.restype = I
    lib.mfa_oracle_e2m1_to_double.argtypes = [ctypes.c_uint8]
    lib.mfa_oracle_e2m1_to_double.restype = ctypes.c_double
    lib.mfa_oracle_e8m0_to_double.argtypes = [ctypes.c_uint8]
    lib.mfa_oracle_e8m0_to_double.restype = ctypes.c_double
    lib.mfa_oracle_e2m1_from_double.argtypes = [ctypes.c_double]
    lib.mfa_oracle_e2m1_from_double.restype = ctypes.c_uint8
    lib.mfa_oracle_mx_block_exponent.argtypes = [P, I]
    lib.mfa_oracle_mx_block_exponent.restype = I
    return lib


KV_FORMATS = {"bf16": 0, "fp8_e4m3": 1, "mxfp4": 2}


def e2m1_to_double(code: int, lib=None) -> float:
    return float((lib or _load()).mfa_oracle_e2m1_to_double(int(code) & 0xF))


def e8m0_to_double(code: int, lib=None) -> float:
    return float((lib or _load()).mfa_oracle_e8m0_to_double(int(code) & 0xFF))


def e2m1_from_double(y: float, lib=None) -> int:
    """Nearest E2M1 code to y (ties to the even code, |y| >= 6 -> 6, sign kept)."""
    return int((lib or _load()).mfa_oracle_e2m1_from_double(float(y)))


def mx_block_exponent(x, lib=None) -> int:
    """OCP MX shared exponent of a block of fp32 values (floor(log2 amax) - 2, in [-127, 127])."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    return int((lib or _load()).mfa_oracle_mx_block_exponent(_ptr(a), a.size))


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = load_library(_LIB)
    return _lib


def num_cpus() -> int:
    return int(_load().mfa_oracle_num_cpus())


def e4m3_to_double(code: int, lib=None) -> float:
    return float((lib or _load()).mfa_oracle_e4m3_to_double(int(code) & 0xFF))


def e4m3_from_float(y: float, lib=None) -> int:
    """Nearest e4m3 code to the fp32 value y (ties to the even code, |y| >= 448 -> 448)."""
    return int((lib or _load()).mfa_oracle_e4m3_from_float(float(y)))


def e4m3_from_float_array(y, lib=None) -> np.ndarray:
    """e4m3_from_float over an fp32 array; returns uint8 codes of the same shape."""
    a = np.ascontiguousarray(np.asarray(y, dtype=np.float32))
    out = np.zeros(a.shape, dtype=np.uint8)
    (lib or _load()).mfa_oracle_e4m3_from_float_array(_ptr(a), a.size, _ptr(out))
    return out


APPEND_BAD_BLOCK = 1      # return-mask bits of kv_append
APPEND_BAD_POSITION = 2


def kv_append(k_new, v_new, positions, block_table, k_cache, v_cache, k_scale=None, v_scale=None,
              page_size: int = 64, tokens_per_seq: int = 1, lib=None):
    """Oracle KV append: returns (k_cache, v_cache, k_scale, v_scale, mask), updated copies.

    k_new/v_new: bf16 [B*T, d] (torch) or uint16 bit arrays, T = tokens_per_seq new rows
    per sequence; positions: int [B], the token index of each sequence's first new row
    (row i goes to positions[b] + i; < 0: none); block_table int32 [B, max_pages];
    caches as produced by the input generator (bf16 [nb, page, d], or uint8 e4m3 codes with
    fp32 scales [nb, page]).  The inputs are not modified.
    """
    kn = np.ascontiguousarray(_np(k_new)).view(np.uint16)
    vn = np.ascontiguousarray(_np(v_new)).view(np.uint16)
    T = int(tokens_per_seq)
    B, d = kn.shape[0] // T, kn.shape[1]
    pos = np.ascontiguousarray(np.asarray(_np(positions), dtype=np.int32))
    table = np.ascontiguousarray(_np(block_table).astype(np.int32))
    kc = np.array(_np(k_cache), copy=True)
    vc = np.array(_np(v_cache), copy=True)
    # the cache format from its layout: bf16 rows, e4m3 rows of d codes, or MXFP4 rows of d/2 bytes
    fmt = 0 if kc.dtype != np.uint8 else (2 if kc.shape[-1] * 2 == d else 1)
    ks = vs = None
    if fmt == 1:
        ks = np.array(_np(k_scale), dtype=np.float32, copy=True)
        vs = np.array(_np(v_scale), dtype=np.float32, copy=True)
    elif fmt == 2:
        ks = np.array(_np(k_scale), dtype=np.uint8, copy=True)
        vs = np.array(_np(v_scale), dtype=np.uint8, copy=True)
    mask = (lib or _load()).mfa_oracle_kv_append(
        B, T, d, page_size, table.shape[1], kc.shape[0], fmt, _ptr(kn), _ptr(vn), _ptr(pos),
        _ptr(table), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs))
    if mask < 0:
        raise ValueError("mfa_oracle_kv_append: bad argument")
    return kc, vc, ks, vs, int(mask)


def _np(t):
    """Contiguous numpy view of a torch CPU tensor (bf16 viewed as uint16)."""
    import torch
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        t = t.contiguous().numpy()
    return np.ascontiguousarray(t)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def decode(case, t_begin=None, t_end=None, nthreads: int = 0,
           softmax_scale: Optional[float] = None, batch_slice: Optional[slice] = None,
           lib=None):
    """Oracle decode of ``case`` -> (out float64 [B*T,H,d], lse float64 [B*T,H]).

    T = case.workload.tokens_per_seq new query tokens per sequence (1: one each).
    case.workload.num_kv_heads = G key/value heads per cache row (query head h reads head
    h // (H // G)); case.workload.kv_shared: the values are the key rows (one latent).

    ``t_begin``/``t_end`` (int sequences of length B) restrict each sequence to
    a token range; ``batch_slice`` restricts the batch (for bounded samples).
    ``lib`` selects another compiled copy of the oracle (mutation tests).
    """
    w = case.workload
    q = _np(case.q)
    table = _np(case.block_table).astype(np.int32)
    lens = _np(case.seq_lens).astype(np.int32)
    T = int(getattr(w, "tokens_per_seq", 1))
    if T > 1:
        # multi-token decode: the T new tokens are the last T cached ones, and query token i
        # of sequence b attends to its cached tokens 0 .. L_b - T + i (causal among the new
        # tokens).  Each (b, i) is then an ordinary decode over b's block-table row.
        i = np.tile(np.arange(T), len(lens))
        table = np.ascontiguousarray(np.repeat(table, T, axis=0))
        lens = np.ascontiguousarray(np.maximum(0, np.repeat(lens, T) - (T - 1 - i)).astype(np.int32))
    if batch_slice is not None:
        q, table, lens = q[batch_slice], table[batch_slice], lens[batch_slice]
        q, table, lens = (np.ascontiguousarray(x) for x in (q, table, lens))
        if t_begin is not None:
            t_begin = np.asarray(t_begin)[batch_slice]
        if t_end is not None:
            t_end = np.asarray(t_end)[batch_slice]
    B, H, d = q.shape
    G = int(getattr(w, "num_kv_heads", 1))
    shared = bool(getattr(w, "kv_shared", False))
    kc = _np(case.k_cache)
    vc = None if shared else _np(case.v_cache)
    ks = _np(case.k_scale)
    vs = None if shared else _np(case.v_scale)
    fmt = KV_FORMATS[w.kv_dtype]
    sdt = np.uint8 if fmt == 2 else np.float32
    if ks is not None:
        ks = np.ascontiguousarray(ks.astype(sdt))
    if vs is not None:
        vs = np.ascontiguousarray(vs.astype(sdt))
    tb = None if t_begin is None else np.ascontiguousarray(np.asarray(t_begin, dtype=np.int32))
    te = None if t_end is None else np.ascontiguousarray(np.asarray(t_end, dtype=np.int32))
    out = np.zeros((B, H, d), dtype=np.float64)
    lse = np.zeros((B, H), dtype=np.float64)
    scale = w.scale() if softmax_scale is None else float(softmax_scale)
    rc = (lib or _load()).mfa_oracle_decode(
        B, H, G, d, w.page_size, table.shape[1], fmt,
        _ptr(q), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(table), _ptr(lens),
        _ptr(tb), _ptr(te), scale, _ptr(out), _ptr(lse), int(nthreads))
    if rc != 0:
        raise ValueError(f"mfa_oracle_decode failed with code {rc}")
    return out, lse


def combine(part_o: np.ndarray, part_lse: np.ndarray):
    """Log-sum-exp merge. part_o [S, ..., d], part_lse [S, ...] -> (out [..., d], lse [...])."""
    part_o = np.ascontiguousarray(part_o, dtype=np.float64)
    part_lse = np.ascontiguousarray(part_lse, dtype=np.float64)
    S = part_o.shape[0]
    d = part_o.shape[-1]
    rest = part_lse.shape[1:]
    R = int(np.prod(rest)) if rest else 1
    out = np.zeros(rest + (d,), dtype=np.float64)
    lse = np.zeros(rest, dtype=np.float64)
    rc = _load().mfa_oracle_combine(S, R, d, _ptr(part_o), _ptr(part_lse), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"mfa_oracle_combine failed with code {rc}")
    return out, lse
