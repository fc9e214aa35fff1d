"""Oracle for batched paged-KV decode attention -- TEST INFRASTRUCTURE ONLY.

A plain f64 CPU restatement of the decode path, written in C (``oxd_oracle.c``)
and loaded here through ctypes. Only ``tests/``, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline leg may use it; the CUDA library never does, and
the two share no code.

What it computes (the definition stated in ``oxd_oracle.h``) follows the
"FlashInfer parity matrix" page, sections "Admitted attention matrix" and
"Domain coverage": one query token per request attends, with full (non-causal)
softmax attention, over the tokens its block table lists, for MHA, GQA and MQA
head groupings, over NHD or HND pages. ``paged_prefill`` restates the same
page's "Paged causal prefill" row: several query tokens per request, the last
of its cached tokens, each attending causally up to its own position.

Inputs are numpy arrays: bf16 tensors as ``uint16`` bit patterns, block tables
as ``int32``. Outputs are float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = [os.path.join(_HERE, "oxd_oracle.c"), os.path.join(_HERE, "oxd_oracle.h")]
_LIB_PATH = os.path.join(_HERE, "liboxd_oracle.so")

LAYOUT_NHD = 0
LAYOUT_HND = 1

_lock = threading.Lock()
_lib = None


def compile_library(src: str, out: str) -> str:
    """gcc build of an oracle source file (C11, -O2, no fast-math, no FMA contraction)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(
        ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
         "-I", _HERE, "-o", tmp, src, "-lm", "-lpthread"],
        check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle if it is missing or older than its sources."""
    stale = force or not os.path.exists(_LIB_PATH) or any(
        os.path.getmtime(s) > os.path.getmtime(_LIB_PATH) for s in _SRC)
    if stale:
        compile_library(_SRC[0], _LIB_PATH)
    return _LIB_PATH


def bind(path: str):
    """Load an oracle build and declare its C signatures."""
    lib = ctypes.CDLL(path)
    p = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_paged_decode_f64.argtypes = [
        i32, i32, i32, i32, i32, i32, i64, p, p, p, p, p, p, f64, p, i32, p, p, i32]
    lib.oracle_paged_decode_f64.restype = i32
    lib.oracle_partial_state_f64.argtypes = [
        i32, i32, i32, i32, i32, i32, i64, p, p, p, p, p, p, f64, i32, i32, i64, i64, p, p]
    lib.oracle_partial_state_f64.restype = i32
    lib.oracle_merge_states_f64.argtypes = [i32, i32, p, p, p, p]
    lib.oracle_merge_states_f64.restype = None
    lib.oracle_paged_prefill_f64.argtypes = [
        i32, i32, i32, i32, i32, i32, i64, p, p, p, p, p, p, p, f64, p, i32, p, p, i32]
    lib.oracle_paged_prefill_f64.restype = i32
    lib.oracle_rope_f64.argtypes = [i32, i32, p, p, f64, p]
    lib.oracle_rope_f64.restype = None
    lib.oracle_f64_to_bf16.argtypes = [f64]
    lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
    lib.oracle_rope_append.argtypes = [i32, i32, i32, i32, i32, i32, i32, i64, p, p, p, p, p, p,
                                       p, p, f64, p, p, p, p]
    lib.oracle_rope_append.restype = i32
    return lib


def _load(lib=None):
    global _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _as(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def _bits(a):
    a = np.asarray(a)
    if a.dtype not in (np.uint16, np.int16):
        raise TypeError("bf16 tensors are passed as uint16/int16 bit patterns")
    return np.ascontiguousarray(a).view(np.uint16)


class OracleError(RuntimeError):
    pass


def paged_decode(q, k_pages, v_pages, indptr, indices, last_page_len, *, num_kv_heads,
                 page_size, layout, sm_scale, heads=None, nthreads=0, lib=None):
    """f64 decode attention.

    q: [B, Hq, D] bf16 bits. k_pages/v_pages: pool of bf16 bits in NHD
    ``[num_pages, page_size, Hkv, D]`` or HND ``[num_pages, Hkv, page_size, D]``.
    heads: optional sequence of (b, hq) pairs; then out is [n, D], lse [n].
    Returns (out, lse) as float64 arrays.
    """
    lib = _load(lib)
    q = _bits(q)
    k = _bits(k_pages)
    v = _bits(v_pages)
    B, Hq, D = q.shape
    indptr = _as(indptr, np.int32)
    indices = _as(indices, np.int32)
    last = _as(last_page_len, np.int32)
    if indptr.shape != (B + 1,) or last.shape != (B,):
        raise ValueError("indptr must be [B+1] and last_page_len [B]")
    per_page = page_size * num_kv_heads * D
    if k.size % per_page or v.size != k.size:
        raise ValueError("K/V pools must hold whole pages of equal count")
    num_pages = k.size // per_page
    if heads is None:
        hl = None
        out = np.empty((B, Hq, D), np.float64)
        lse = np.empty((B, Hq), np.float64)
        n = B * Hq
    else:
        hl = _as(heads, np.int32).reshape(-1, 2)
        n = hl.shape[0]
        out = np.empty((n, D), np.float64)
        lse = np.empty((n,), np.float64)
    rc = lib.oracle_paged_decode_f64(
        B, Hq, num_kv_heads, D, page_size, layout, num_pages, _ptr(q), _ptr(k), _ptr(v),
        _ptr(indptr), _ptr(indices), _ptr(last), float(sm_scale),
        None if hl is None else _ptr(hl), n, _ptr(out), _ptr(lse), int(nthreads))
    if rc != 0:
        raise OracleError(f"oracle_paged_decode_f64 returned {rc}")
    return out, lse


def paged_prefill(q, k_pages, v_pages, qo_indptr, indptr, indices, last_page_len, *,
                  num_kv_heads, page_size, layout, sm_scale, rows=None, nthreads=0, lib=None):
    """f64 causal prefill attention over paged KV.

    q: [Nq, Hq, D] bf16 bits, Nq = qo_indptr[-1]; request b's query tokens are
    its last qo_indptr[b+1] - qo_indptr[b] cached tokens. Pools and block
    tables as for ``paged_decode``. rows: optional sequence of (token, hq)
    pairs; then out is [n, D], lse [n]. Returns (out, lse) as float64 arrays.
    """
    lib = _load(lib)
    q = _bits(q)
    k = _bits(k_pages)
    v = _bits(v_pages)
    Nq, Hq, D = q.shape
    qo = _as(qo_indptr, np.int32)
    indptr = _as(indptr, np.int32)
    indices = _as(indices, np.int32)
    last = _as(last_page_len, np.int32)
    B = last.shape[0]
    if indptr.shape != (B + 1,) or qo.shape != (B + 1,) or int(qo[-1]) != Nq:
        raise ValueError("qo_indptr and indptr must be [B+1], qo_indptr[B] = q.shape[0]")
    per_page = page_size * num_kv_heads * D
    if k.size % per_page or v.size != k.size:
        raise ValueError("K/V pools must hold whole pages of equal count")
    num_pages = k.size // per_page
    if rows is None:
        rl = None
        out = np.empty((Nq, Hq, D), np.float64)
        lse = np.empty((Nq, Hq), np.float64)
        n = Nq * Hq
    else:
        rl = _as(rows, np.int32).reshape(-1, 2)
        n = rl.shape[0]
        out = np.empty((n, D), np.float64)
        lse = np.empty((n,), np.float64)
    rc = lib.oracle_paged_prefill_f64(
        B, Hq, num_kv_heads, D, page_size, layout, num_pages, _ptr(q), _ptr(k), _ptr(v),
        _ptr(qo), _ptr(indptr), _ptr(indices), _ptr(last), float(sm_scale),
        None if rl is None else _ptr(rl), n, _ptr(out), _ptr(lse), int(nthreads))
    if rc != 0:
        raise OracleError(f"oracle_paged_prefill_f64 returned {rc}")
    return out, lse


def partial_state(q, k_pages, v_pages, indptr, indices, last_page_len, *, num_kv_heads,
                  page_size, layout, sm_scale, b, hq, tok_begin, tok_end, lib=None):
    """State (o[D], lse) of head (b, hq) over logical tokens [tok_begin, tok_end)."""
    lib = _load(lib)
    q = _bits(q)
    k = _bits(k_pages)
    v = _bits(v_pages)
    B, Hq, D = q.shape
    indptr = _as(indptr, np.int32)
    indices = _as(indices, np.int32)
    last = _as(last_page_len, np.int32)
    num_pages = k.size // (page_size * num_kv_heads * D)
    o = np.empty((D,), np.float64)
    lse = np.empty((1,), np.float64)
    rc = lib.oracle_partial_state_f64(
        B, Hq, num_kv_heads, D, page_size, layout, num_pages, _ptr(q), _ptr(k), _ptr(v),
        _ptr(indptr), _ptr(indices), _ptr(last), float(sm_scale), int(b), int(hq),
        int(tok_begin), int(tok_end), _ptr(o), _ptr(lse))
    if rc != 0:
        raise OracleError(f"oracle_partial_state_f64 returned {rc}")
    return o, float(lse[0])


def merge_states(v, s, lib=None):
    """Merge S states of one head: v [S, D] float64, s [S] float64 -> (out [D], lse)."""
    lib = _load(lib)
    v = _as(v, np.float64)
    s = _as(s, np.float64)
    S, D = v.shape
    out = np.empty((D,), np.float64)
    lse = np.empty((1,), np.float64)
    lib.oracle_merge_states_f64(S, D, _ptr(v), _ptr(s), _ptr(out), _ptr(lse))
    return out, float(lse[0])


def merge_states_batched(v, s):
    """Merge over axis 1: v [N, S, H, D], s [N, S, H] -> (out [N, H, D], lse [N, H])."""
    v = _as(v, np.float64)
    s = _as(s, np.float64)
    N, S, H, D = v.shape
    out = np.empty((N, H, D), np.float64)
    lse = np.empty((N, H), np.float64)
    for n in range(N):
        for h in range(H):
            out[n, h], lse[n, h] = merge_states(v[n, :, h, :], s[n, :, h])
    return out, lse


# ------------------------------------------------------------------ RoPE and paged append

APPEND_WRITTEN = 0
APPEND_SHARED_PAGE = 1
APPEND_BAD_POSITION = 2
APPEND_BAD_PAGE = 3


def rope(x, positions, theta=10000.0, lib=None):
    """f64 split-half rotary embedding of the rows of x ([n, D] float64) at
    positions ([n] int32); returns [n, D] float64 (see ``oxd_oracle.h``)."""
    L = _load(lib)
    x = _as(x, np.float64)
    n, D = x.shape
    pos = _as(positions, np.int32)
    if pos.shape != (n,):
        raise ValueError("one position per row")
    y = np.empty_like(x)
    L.oracle_rope_f64(n, D, _ptr(x), _ptr(pos), float(theta), _ptr(y))
    return y


def f64_to_bf16(x, lib=None):
    """Nearest bfloat16 (ties to even) of each element, as uint16 bit patterns."""
    L = _load(lib)
    a = np.asarray(x, np.float64)
    return np.array([L.oracle_f64_to_bf16(float(v)) for v in a.ravel()],
                    np.uint16).reshape(a.shape)


def rope_append(q, k, v, token_request, positions, indptr, indices, refcount, k_pages,
                v_pages, *, page_size, layout, theta=10000.0, lib=None):
    """Fused RoPE + paged append on copies of the pools.

    q: [T, Hq, D], k, v: [T, Hkv, D] bf16 bits; pools as for ``paged_decode``.
    Returns (q_out bits, k_pages bits, v_pages bits, status [T] int32)."""
    L = _load(lib)
    q, k, v = _bits(q), _bits(k), _bits(v)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    kp, vp = _bits(k_pages).copy(), _bits(v_pages).copy()
    num_pages = kp.shape[0]
    indptr = _as(indptr, np.int32)
    B = indptr.shape[0] - 1
    tr, pos = _as(token_request, np.int32), _as(positions, np.int32)
    idx, rc = _as(indices, np.int32), _as(refcount, np.int32)
    q_out = np.empty_like(q)
    status = np.empty(T, np.int32)
    r = L.oracle_rope_append(T, B, Hq, Hkv, D, page_size, layout, num_pages, _ptr(q), _ptr(k),
                             _ptr(v), _ptr(tr), _ptr(pos), _ptr(indptr), _ptr(idx), _ptr(rc),
                             float(theta), _ptr(q_out), _ptr(kp), _ptr(vp), _ptr(status))
    if r < 0:
        raise OracleError(f"oracle_rope_append failed ({r})")
    return q_out, kp, vp, status
