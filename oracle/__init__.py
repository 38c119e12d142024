"""Python access to the plain fp64 CPU oracle for QSA block-sparse GQA.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers.  The oracle shares no code
with the CUDA library (``block_sparse_gqa_qsa_gb300``) and never imports it;
the CUDA path never imports this package.

Arrays are numpy; fp16 tensors are passed as ``np.float16`` (their bits go
through unchanged).  Every wrapper checks the return code and raises
``ValueError`` on invalid arguments.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsa_oracle.cpp")
_HDR = os.path.join(_HERE, "qsa_oracle.h")
_LIB = os.path.join(_HERE, "libqsa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host C++ compiler (no CUDA involved)."""
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest_src:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-Wall", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            vp = ctypes.c_void_p
            L.qsa_oracle_half_to_double.argtypes = [ctypes.c_uint16]
            L.qsa_oracle_half_to_double.restype = dbl
            L.qsa_oracle_double_to_half.argtypes = [dbl]
            L.qsa_oracle_double_to_half.restype = ctypes.c_uint16
            L.qsa_oracle_index_q.argtypes = [vp, vp, i32, i32, i64, dbl, dbl, vp]
            L.qsa_oracle_index_q.restype = i32
            L.qsa_oracle_block_key.argtypes = [vp, i32, vp, i32, i32, i64, dbl, dbl, vp, vp]
            L.qsa_oracle_block_key.restype = i32
            L.qsa_oracle_block_score.argtypes = [vp, vp, i32, i32]
            L.qsa_oracle_block_score.restype = dbl
            L.qsa_oracle_select.argtypes = [vp, i32, i32, vp]
            L.qsa_oracle_select.restype = i32
            L.qsa_oracle_expand.argtypes = [vp, i32, i32, i64, i32, i32, vp]
            L.qsa_oracle_expand.restype = i32
            L.qsa_oracle_indexer_prefill.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                                     i32, i32, dbl, dbl, vp, i64, vp, vp, vp, i32]
            L.qsa_oracle_indexer_prefill.restype = i32
            L.qsa_oracle_sparse_prefill.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                                    dbl, vp, i64, vp, i32]
            L.qsa_oracle_sparse_prefill.restype = i32
            L.qsa_oracle_indexer_decode_state.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, i32, i32,
                                                          i32, i32, i32, dbl, dbl, vp, vp, vp]
            L.qsa_oracle_indexer_decode_state.restype = i32
            L.qsa_oracle_indexer_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                    i32, i32, i32, i32, i32, i32, i32, dbl, dbl, vp, vp,
                                                    i32]
            L.qsa_oracle_indexer_decode.restype = i32
            L.qsa_oracle_attend_rows.argtypes = [vp, vp, vp, i64, i32, i32, i32, dbl, vp]
            L.qsa_oracle_attend_rows.restype = i32
            L.qsa_oracle_sparse_decode.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                                   i32, dbl, vp, i32]
            L.qsa_oracle_sparse_decode.restype = i32
            L.qsa_oracle_sparse_prefill_bf16.argtypes = L.qsa_oracle_sparse_prefill.argtypes
            L.qsa_oracle_sparse_prefill_bf16.restype = i32
            L.qsa_oracle_attend_rows_bf16.argtypes = L.qsa_oracle_attend_rows.argtypes
            L.qsa_oracle_attend_rows_bf16.restype = i32
            L.qsa_oracle_sparse_decode_bf16.argtypes = L.qsa_oracle_sparse_decode.argtypes
            L.qsa_oracle_sparse_decode_bf16.restype = i32
            L.qsa_oracle_rope_qkv.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, dbl, dbl, vp, vp, vp,
                                              i32]
            L.qsa_oracle_rope_qkv.restype = i32
            L.qsa_oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.qsa_oracle_bf16_to_double.restype = dbl
            _lib = L
    return _lib


def _arr(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _opt(a, dtype):
    if a is None:
        return None, None
    return _arr(a, dtype)


def _check(rc, what):
    if rc < 0:
        raise ValueError(f"oracle {what}: invalid arguments (rc={rc})")
    return rc


# ---------------------------------------------------------------- fp16 bits
def bf16_to_double(bits: int) -> float:
    return lib().qsa_oracle_bf16_to_double(bits)


def half_to_double(bits: int) -> float:
    return lib().qsa_oracle_half_to_double(int(bits) & 0xFFFF)


def double_to_half(x: float) -> int:
    return lib().qsa_oracle_double_to_half(float(x))


# ----------------------------------------------------------- indexer steps
def index_q(x, w, rot, pos, theta, eps):
    """RMSNorm*(1+w) + partial RoPE at ``pos`` of one fp16 vector -> f64."""
    x, xp = _arr(x, np.float16)
    w, wp = _arr(w, np.float32)
    y = np.zeros(x.shape[-1], np.float64)
    _check(lib().qsa_oracle_index_q(xp, wp, x.shape[-1], rot, int(pos), theta, eps,
                                    y.ctypes.data_as(ctypes.c_void_p)), "index_q")
    return y


def block_key(raw, w, rot, pos, theta, eps):
    """Block key of ``raw`` (fp16 [r, di]); returns (fp16 kbar, f64 value before rounding)."""
    raw, rp = _arr(raw, np.float16)
    w, wp = _arr(w, np.float32)
    r, di = raw.shape
    kb = np.zeros(di, np.float16)
    y = np.zeros(di, np.float64)
    _check(lib().qsa_oracle_block_key(rp, r, wp, di, rot, int(pos), theta, eps,
                                      kb.ctypes.data_as(ctypes.c_void_p),
                                      y.ctypes.data_as(ctypes.c_void_p)), "block_key")
    return kb, y


def block_score(q, kbar):
    q, qp = _arr(q, np.float64)
    kbar, kp = _arr(kbar, np.float16)
    Hi, di = q.shape
    return lib().qsa_oracle_block_score(qp, kp, Hi, di)


def select(scores, budget):
    s, sp = _arr(scores, np.float64)
    sel = np.zeros(max(len(s), 1), np.int32)
    n = _check(lib().qsa_oracle_select(sp, len(s), budget, sel.ctypes.data_as(ctypes.c_void_p)),
               "select")
    return sel[:n]


def expand(sel, n_c, t, ratio, topK):
    sel, selp = _arr(sel, np.int32)
    out = np.zeros(topK, np.int32)
    _check(lib().qsa_oracle_expand(selp, len(sel), n_c, int(t), ratio, topK,
                                   out.ctypes.data_as(ctypes.c_void_p)), "expand")
    return out


# ------------------------------------------------------------ whole passes
def indexer_prefill(idxQ, idxK, wq, wk, ctx, *, rot, ratio, budget, topK, theta, eps,
                    rows=None, want_kbar=False, want_scores=False, nthreads=0):
    """Index lists for all rows (``rows=None``) or for the flat rows ``b*S+t`` given.

    Returns ``indices`` ([B,S,topK] or [len(rows),topK]) and, when asked,
    ``kbar`` fp16 [B,S//ratio,di] and ``scores`` f64 [nrows,S//ratio].
    """
    idxQ, qp = _arr(idxQ, np.float16)
    idxK, kp = _arr(idxK, np.float16)
    wq, wqp = _arr(wq, np.float32)
    wk, wkp = _arr(wk, np.float32)
    ctx, cp = _arr(ctx, np.int32)
    B, S, Hi, di = idxQ.shape
    rows_a, rp = _opt(rows, np.int64)
    nrows = B * S if rows is None else len(rows_a)
    ind = np.empty((nrows, topK), np.int32)
    kbar = np.zeros((B, S // ratio, di), np.float16) if want_kbar else None
    sc = np.empty((nrows, S // ratio), np.float64) if want_scores else None
    _check(lib().qsa_oracle_indexer_prefill(
        qp, kp, wqp, wkp, cp, B, S, Hi, di, rot, ratio, budget, topK, theta, eps, rp,
        nrows, ind.ctypes.data_as(ctypes.c_void_p),
        None if kbar is None else kbar.ctypes.data_as(ctypes.c_void_p),
        None if sc is None else sc.ctypes.data_as(ctypes.c_void_p), nthreads), "indexer_prefill")
    if rows is None:
        ind = ind.reshape(B, S, topK)
    out = [ind]
    if want_kbar:
        out.append(kbar)
    if want_scores:
        out.append(sc)
    return out[0] if len(out) == 1 else tuple(out)


def sparse_prefill(q, k, v, indices, ctx, scale, rows=None, nthreads=0, bf16=False):
    """f64 attention output ([B,S,Hq,D], or [len(rows),Hq,D] with row-compact indices).
    bf16=True: q/k/v are bfloat16 bit patterns (np.uint16)."""
    et = np.uint16 if bf16 else np.float16
    q, qp = _arr(q, et)
    k, kp = _arr(k, et)
    v, vp = _arr(v, et)
    ctx, cp = _arr(ctx, np.int32)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    indices, ip = _arr(indices, np.int32)
    topK = indices.shape[-1]
    rows_a, rp = _opt(rows, np.int64)
    nrows = B * S if rows is None else len(rows_a)
    out = np.empty((nrows, Hq, D), np.float64)
    fn = lib().qsa_oracle_sparse_prefill_bf16 if bf16 else lib().qsa_oracle_sparse_prefill
    rc = fn(qp, kp, vp, ip, cp, B, S, Hq, Hkv, D, topK, scale, rp, nrows, out.ctypes.data_as(ctypes.c_void_p),
            nthreads)
    if rc == -2:
        raise ValueError("oracle sparse_prefill: an index list names a token at or past the live length")
    _check(rc, "sparse_prefill")
    return out.reshape(B, S, Hq, D) if rows is None else out


def indexer_decode_state(idxQ, idxK, wq, wk, kbar, tail, L, *, rot, ratio, budget, topK, theta, eps):
    """Decode indexer of one sequence from compact state; returns (indices, kbar_new|None, scores)."""
    idxQ, qp = _arr(idxQ, np.float16)
    idxK, kp = _arr(idxK, np.float16)
    wq, wqp = _arr(wq, np.float32)
    wk, wkp = _arr(wk, np.float32)
    Hi, di = idxQ.shape
    kbar, kbp = _opt(kbar, np.float16)
    tail, tp = _opt(tail, np.float16)
    ind = np.empty(topK, np.int32)
    knew = np.zeros(di, np.float16)
    sc = np.empty(max(L // ratio, 1), np.float64)
    rc = _check(lib().qsa_oracle_indexer_decode_state(
        qp, kp, wqp, wkp, kbp, tp, int(L), Hi, di, rot, ratio, budget, topK, theta, eps,
        ind.ctypes.data_as(ctypes.c_void_p), knew.ctypes.data_as(ctypes.c_void_p),
        sc.ctypes.data_as(ctypes.c_void_p)), "indexer_decode_state")
    return ind, (knew if rc == 1 else None), sc[: L // ratio]


def indexer_decode(idxQ, idxK, wq, wk, pool, page_table, ctx, *, D, rot, ratio, budget, topK, theta,
                   eps, want_scores=False, nthreads=0):
    """Decode indexer over the paged pool; ``pool`` (np.float16) is updated in place."""
    idxQ, qp = _arr(idxQ, np.float16)
    idxK, kp = _arr(idxK, np.float16)
    wq, wqp = _arr(wq, np.float32)
    wk, wkp = _arr(wk, np.float32)
    if pool.dtype != np.float16 or not pool.flags["C_CONTIGUOUS"]:
        raise ValueError("pool must be a C-contiguous float16 array (updated in place)")
    page_table, ptp = _arr(page_table, np.int32)
    ctx, cp = _arr(ctx, np.int32)
    B, Hi, di = idxQ.shape
    numFlatPages, tpp, Hkv, poolHeadDim = pool.shape
    maxPages = page_table.shape[-1]
    ind = np.empty((B, topK), np.int32)
    nbmax = maxPages * tpp // ratio
    sc = np.empty((B, nbmax), np.float64) if want_scores else None
    _check(lib().qsa_oracle_indexer_decode(
        qp, kp, wqp, wkp, pool.ctypes.data_as(ctypes.c_void_p), ptp, cp, B, Hkv, D, poolHeadDim,
        numFlatPages, maxPages, Hi, di, rot, ratio, budget, topK, theta, eps,
        ind.ctypes.data_as(ctypes.c_void_p), None if sc is None else sc.ctypes.data_as(ctypes.c_void_p),
        nthreads), "indexer_decode")
    return (ind, sc) if want_scores else ind


def attend_rows(q, krows, vrows, scale, bf16=False):
    """Attention of one token (q [Hq,D]) over gathered rows ([n,Hkv,D]) -> f64 [Hq,D]; fp16, or bfloat16
    bit patterns (np.uint16) with bf16=True."""
    et = np.uint16 if bf16 else np.float16
    q, qp = _arr(q, et)
    krows, kp = _arr(krows, et)
    vrows, vp = _arr(vrows, et)
    Hq, D = q.shape
    n, Hkv, _ = krows.shape
    out = np.empty((Hq, D), np.float64)
    fn = lib().qsa_oracle_attend_rows_bf16 if bf16 else lib().qsa_oracle_attend_rows
    _check(fn(qp, kp, vp, n, Hq, Hkv, D, scale, out.ctypes.data_as(ctypes.c_void_p)), "attend_rows")
    return out


def sparse_decode(q, pool, page_table, indices, ctx, *, D, scale, nthreads=0, bf16=False):
    """Decode attention over the paged pool -> f64 [B,Hq,D]; bf16=True: q and pool are bfloat16 bit
    patterns (np.uint16)."""
    et = np.uint16 if bf16 else np.float16
    q, qp = _arr(q, et)
    pool, pp = _arr(pool, et)
    page_table, ptp = _arr(page_table, np.int32)
    indices, ip = _arr(indices, np.int32)
    ctx, cp = _arr(ctx, np.int32)
    B, Hq, _ = q.shape
    numFlatPages, _, Hkv, poolHeadDim = pool.shape
    maxPages = page_table.shape[-1]
    topK = indices.shape[-1]
    out = np.empty((B, Hq, D), np.float64)
    fn = lib().qsa_oracle_sparse_decode_bf16 if bf16 else lib().qsa_oracle_sparse_decode
    rc = fn(qp, pp, ptp, ip, cp, B, Hq, Hkv, D, poolHeadDim, numFlatPages, maxPages, topK, scale,
            out.ctypes.data_as(ctypes.c_void_p), nthreads)
    if rc == -2:
        raise ValueError("oracle sparse_decode: an index list names a token at or past the live length")
    _check(rc, "sparse_decode")
    return out


def rope_qkv(qkv, qw, kw, ctx, *, Hq, Hkv, rot, theta, eps, nthreads=0):
    """Upstream q/k norm + partial RoPE of packed QKV fp16 [B,S,Hq+2Hkv,D] -> (q [B,S,Hq,D], k, v [B,S,Hkv,D]),
    fp16 rounded once from f64."""
    qkv, xp = _arr(qkv, np.float16)
    qw, qwp = _arr(qw, np.float32)
    kw, kwp = _arr(kw, np.float32)
    ctx, cp = _arr(ctx, np.int32)
    B, S, NH, D = qkv.shape
    if NH != Hq + 2 * Hkv:
        raise ValueError("rope_qkv: head count mismatch")
    q = np.empty((B, S, Hq, D), np.float16)
    k = np.empty((B, S, Hkv, D), np.float16)
    v = np.empty((B, S, Hkv, D), np.float16)
    _check(lib().qsa_oracle_rope_qkv(xp, qwp, kwp, cp, B, S, Hq, Hkv, D, rot, theta, eps,
                                     q.ctypes.data_as(ctypes.c_void_p), k.ctypes.data_as(ctypes.c_void_p),
                                     v.ctypes.data_as(ctypes.c_void_p), nthreads), "rope_qkv")
    return q, k, v
