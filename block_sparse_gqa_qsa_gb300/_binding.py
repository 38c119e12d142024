"""ctypes binding of libqsa.so (the C ABI declared in include/qsa.h).

Argument marshalling only: every function checks dtypes, devices and
contiguity of torch tensors, fills the C params struct and calls the entry
point of the same name; all computation happens in the library's kernels.
A non-QSA_OK status raises ``QsaError`` with the library's message.  There is
no CPU fallback: a missing library raises ``RuntimeError`` on first use.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqsa.so")

QSA_OK, QSA_ERR_INVALID_ARG, QSA_ERR_UNSUPPORTED, QSA_ERR_WORKSPACE, QSA_ERR_CUDA = range(5)

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_f32 = ctypes.c_float
_sz = ctypes.c_size_t


class QsaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_names.get(status, status)}: {message}")
        self.status = status


_status_names = {0: "QSA_OK", 1: "QSA_ERR_INVALID_ARG", 2: "QSA_ERR_UNSUPPORTED", 3: "QSA_ERR_WORKSPACE",
                 4: "QSA_ERR_CUDA"}


class QsaIndexerPrefillParams(ctypes.Structure):
    _fields_ = [("idxQ", _vp), ("idxK", _vp), ("qNormW", _vp), ("kNormW", _vp), ("contextLengths", _vp),
                ("indices", _vp), ("workspace", _vp), ("workspaceBytes", _sz), ("batchSize", _i32),
                ("seqLen", _i32), ("numHeads", _i32), ("headDim", _i32), ("rotDim", _i32),
                ("compressRatio", _i32), ("budget", _i32), ("topK", _i32), ("ropeTheta", _f32),
                ("rmsNormEps", _f32), ("stream", _vp)]


class QsaIndexerDecodeParams(ctypes.Structure):
    _fields_ = [("idxQ", _vp), ("idxK", _vp), ("qNormW", _vp), ("kNormW", _vp), ("kvPool", _vp),
                ("pageTable", _vp), ("contextLengths", _vp), ("indices", _vp), ("workspace", _vp),
                ("workspaceBytes", _sz), ("batchSize", _i32), ("numKVHeads", _i32), ("kvHeadDim", _i32),
                ("poolHeadDim", _i32), ("numFlatPages", _i32), ("maxPagesPerSeq", _i32), ("numHeads", _i32),
                ("headDim", _i32), ("rotDim", _i32), ("compressRatio", _i32), ("budget", _i32), ("topK", _i32),
                ("ropeTheta", _f32), ("rmsNormEps", _f32), ("stream", _vp)]


class QsaIndexerHandoffParams(ctypes.Structure):
    _fields_ = [("idxK", ctypes.c_void_p), ("contextLengths", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspaceBytes", ctypes.c_size_t), ("kvPool", ctypes.c_void_p), ("pageTable", ctypes.c_void_p),
                ("batchSize", _i32), ("seqLen", _i32), ("headDim", _i32), ("compressRatio", _i32),
                ("numKVHeads", _i32), ("kvHeadDim", _i32), ("poolHeadDim", _i32), ("numFlatPages", _i32),
                ("maxPagesPerSeq", _i32), ("stream", ctypes.c_void_p)]


class QsaRopeQkvParams(ctypes.Structure):
    _fields_ = [("qkv", ctypes.c_void_p), ("qNormW", ctypes.c_void_p), ("kNormW", ctypes.c_void_p),
                ("contextLengths", ctypes.c_void_p), ("qOut", ctypes.c_void_p), ("kOut", ctypes.c_void_p),
                ("vOut", ctypes.c_void_p), ("kvPool", ctypes.c_void_p), ("pageTable", ctypes.c_void_p),
                ("batchSize", _i32), ("seqLen", _i32), ("numQHeads", _i32), ("numKVHeads", _i32),
                ("headDim", _i32), ("rotDim", _i32), ("poolHeadDim", _i32), ("numFlatPages", _i32),
                ("maxPagesPerSeq", _i32), ("ropeTheta", ctypes.c_float), ("rmsNormEps", ctypes.c_float),
                ("stream", ctypes.c_void_p)]


class QsaSparsePrefillParams(ctypes.Structure):
    _fields_ = [("qPtr", _vp), ("kPtr", _vp), ("vPtr", _vp), ("oPtr", _vp), ("indices", _vp),
                ("contextLengths", _vp), ("batchSize", _i32), ("seqLen", _i32), ("numQHeads", _i32),
                ("numKVHeads", _i32), ("headDim", _i32), ("topK", _i32), ("attentionScale", _f32),
                ("stream", _vp), ("status", _vp)]


class QsaSparseDecodeParams(ctypes.Structure):
    _fields_ = [("qPtr", _vp), ("kvPoolPtr", _vp), ("pageTable", _vp), ("indices", _vp),
                ("contextLengths", _vp), ("oPtr", _vp), ("partialO", _vp), ("partialStats", _vp),
                ("splitCounters", _vp), ("batchSize", _i32), ("numQHeads", _i32), ("numKVHeads", _i32),
                ("headDim", _i32), ("poolHeadDim", _i32), ("numFlatPages", _i32), ("maxPagesPerSeq", _i32),
                ("topK", _i32), ("attentionScale", _f32), ("stream", _vp), ("status", _vp)]


class QsaGatherParams(ctypes.Structure):
    _fields_ = [("kvPool", _vp), ("pageTable", _vp), ("indices", _vp), ("contextLengths", _vp), ("scratch", _vp),
                ("scratchPageTable", _vp), ("scratchIndices", _vp), ("scratchLengths", _vp), ("batchSize", _i32),
                ("numKVHeads", _i32), ("headDim", _i32), ("poolHeadDim", _i32), ("numFlatPages", _i32),
                ("maxPagesPerSeq", _i32), ("topK", _i32), ("stream", _vp)]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises RuntimeError when it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libqsa.so is missing ({LIB_PATH}); build it with "
                                   "`python -m block_sparse_gqa_qsa_gb300.build` -- there is no fallback")
            L = ctypes.CDLL(LIB_PATH)
            for name, st in (("qsa_indexer_prefill", QsaIndexerPrefillParams),
                             ("qsa_indexer_decode", QsaIndexerDecodeParams),
                             ("qsa_sparse_prefill", QsaSparsePrefillParams),
                             ("qsa_sparse_decode", QsaSparseDecodeParams),
                             ("qsa_sparse_decode_noalloc", QsaSparseDecodeParams),
                             ("qsa_indexer_prefill_handoff", QsaIndexerHandoffParams),
                             ("qsa_sparse_prefill_bf16", QsaSparsePrefillParams),
                             ("qsa_sparse_prefill_tcgen05", QsaSparsePrefillParams),
                             ("qsa_sparse_prefill_tcgen05_bf16", QsaSparsePrefillParams),
                             ("qsa_sparse_decode_bf16", QsaSparseDecodeParams),
                             ("qsa_rope_qkv", QsaRopeQkvParams),
                             ("qsa_gather_selected", QsaGatherParams)):
                f = getattr(L, name)
                f.argtypes = [ctypes.POINTER(st)]
                f.restype = ctypes.c_int
            L.qsa_indexer_prefill_workspace_size.argtypes = [_i32] * 4
            L.qsa_indexer_prefill_workspace_size.restype = _sz
            L.qsa_indexer_decode_workspace_size.argtypes = [_i32] * 4
            L.qsa_indexer_decode_workspace_size.restype = _sz
            L.qsa_sparse_decode_partial_o_elems.argtypes = [_i32] * 3
            L.qsa_sparse_decode_partial_o_elems.restype = _sz
            L.qsa_sparse_decode_partial_stats_elems.argtypes = [_i32] * 2
            L.qsa_sparse_decode_partial_stats_elems.restype = _sz
            L.qsa_sparse_decode_counter_elems.argtypes = [_i32] * 2
            L.qsa_sparse_decode_counter_elems.restype = _sz
            L.qsa_gather_scratch_elems.argtypes = [_i32] * 4
            L.qsa_gather_scratch_elems.restype = _sz
            L.qsa_gather_scratch_pages.argtypes = [_i32]
            L.qsa_gather_scratch_pages.restype = _i32
            for n in ("qsa_sparse_decode_max_splits", "qsa_sparse_decode_partial_rows",
                      "qsa_indexer_prefill_max_blocks", "qsa_indexer_prefill_max_seq_len"):
                getattr(L, n).argtypes = []
                getattr(L, n).restype = _i32
            L.qsa_sparse_prefill_can_implement.argtypes = [_i32] * 3
            L.qsa_sparse_prefill_can_implement.restype = _i32
            L.qsa_sparse_decode_can_implement.argtypes = [_i32] * 4
            L.qsa_sparse_decode_can_implement.restype = _i32
            L.qsa_status_string.argtypes = [ctypes.c_int]
            L.qsa_status_string.restype = ctypes.c_char_p
            L.qsa_last_error_message.argtypes = []
            L.qsa_last_error_message.restype = ctypes.c_char_p
            L.qsa_last_device_error.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(_i32)]
            L.qsa_last_device_error.restype = ctypes.c_int
            L.qsa_debug_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            L.qsa_debug_set_wait_limit_ns.restype = None
            _lib = L
    return _lib


def _check(status: int) -> None:
    if status != QSA_OK:
        raise QsaError(status, lib().qsa_last_error_message().decode())


def _ptr(t: torch.Tensor | None, dtype=None, name: str = "tensor") -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ------------------------------------------------------------------ sizes
def indexer_prefill_workspace_size(B: int, S: int, di: int, ratio: int) -> int:
    return lib().qsa_indexer_prefill_workspace_size(B, S, di, ratio)


def indexer_decode_workspace_size(B: int, max_pages_per_seq: int, ratio: int, budget: int) -> int:
    return lib().qsa_indexer_decode_workspace_size(B, max_pages_per_seq, ratio, budget)


def sparse_decode_workspace_elems(B: int, Hkv: int, D: int) -> tuple[int, int, int]:
    L = lib()
    return (L.qsa_sparse_decode_partial_o_elems(B, Hkv, D), L.qsa_sparse_decode_partial_stats_elems(B, Hkv),
            L.qsa_sparse_decode_counter_elems(B, Hkv))


def debug_set_wait_limit_ns(ns: int) -> None:
    """qsa_debug_set_wait_limit_ns: a test bound on the decode scorer's progress waits (0 restores 0.2 s)."""
    lib().qsa_debug_set_wait_limit_ns(int(ns))


def last_device_error(workspace: torch.Tensor, stream=None) -> int:
    """The status word of an indexer workspace (device-side error bits); waits for `stream`."""
    out = _i32(0)
    _check(lib().qsa_last_device_error(_ptr(workspace, name="workspace"), _stream(stream), ctypes.byref(out)))
    st = stream if stream is not None else torch.cuda.current_stream()
    if hasattr(st, "synchronize"):
        st.synchronize()
    else:
        torch.cuda.synchronize()
    return int(out.value)


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Zero-filled byte buffer (torch allocations are 256-byte aligned)."""
    return torch.zeros(max(nbytes, 1), dtype=torch.uint8, device=device)


# ------------------------------------------------------------- entry points
def indexer_prefill(idxQ, idxK, wq, wk, ctx, indices, workspace, *, rot, ratio, budget, topK, theta, eps,
                    stream=None):
    """qsa_indexer_prefill: idxQ fp16 [B,S,Hi,di], idxK fp16 [B,S,di] -> indices int32 [B,S,topK]."""
    B, S, Hi, di = idxQ.shape
    p = QsaIndexerPrefillParams(
        idxQ=_ptr(idxQ, torch.float16, "idxQ"), idxK=_ptr(idxK, torch.float16, "idxK"),
        qNormW=_ptr(wq, torch.float32, "qNormW"), kNormW=_ptr(wk, torch.float32, "kNormW"),
        contextLengths=_ptr(ctx, torch.int32, "contextLengths"), indices=_ptr(indices, torch.int32, "indices"),
        workspace=_ptr(workspace, None, "workspace"), workspaceBytes=workspace.numel() * workspace.element_size(),
        batchSize=B, seqLen=S, numHeads=Hi, headDim=di, rotDim=rot, compressRatio=ratio, budget=budget,
        topK=topK, ropeTheta=theta, rmsNormEps=eps, stream=_stream(stream))
    if tuple(idxK.shape) != (B, S, di) or tuple(indices.shape[-1:]) != (topK,) or indices.numel() != B * S * topK:
        raise ValueError("indexer_prefill: shape mismatch")
    _check(lib().qsa_indexer_prefill(ctypes.byref(p)))


def indexer_decode(idxQ, idxK, wq, wk, pool, page_table, ctx, indices, workspace, *, D, rot, ratio, budget,
                   topK, theta, eps, stream=None):
    """qsa_indexer_decode: one new token per sequence; updates the pool's tail state in place."""
    B, Hi, di = idxQ.shape
    nflat, tpp, Hkv, phd = pool.shape
    p = QsaIndexerDecodeParams(
        idxQ=_ptr(idxQ, torch.float16, "idxQ"), idxK=_ptr(idxK, torch.float16, "idxK"),
        qNormW=_ptr(wq, torch.float32, "qNormW"), kNormW=_ptr(wk, torch.float32, "kNormW"),
        kvPool=_ptr(pool, torch.float16, "kvPool"), pageTable=_ptr(page_table, torch.int32, "pageTable"),
        contextLengths=_ptr(ctx, torch.int32, "contextLengths"), indices=_ptr(indices, torch.int32, "indices"),
        workspace=_ptr(workspace, None, "workspace"), workspaceBytes=workspace.numel() * workspace.element_size(),
        batchSize=B, numKVHeads=Hkv, kvHeadDim=D, poolHeadDim=phd, numFlatPages=nflat,
        maxPagesPerSeq=page_table.shape[-1], numHeads=Hi, headDim=di, rotDim=rot, compressRatio=ratio,
        budget=budget, topK=topK, ropeTheta=theta, rmsNormEps=eps, stream=_stream(stream))
    if tpp != 128 or tuple(page_table.shape[:2]) != (B, 2) or indices.numel() != B * topK:
        raise ValueError("indexer_decode: shape mismatch")
    _check(lib().qsa_indexer_decode(ctypes.byref(p)))


def indexer_prefill_handoff(idxK, ctx, workspace, pool, page_table, *, D, ratio, stream=None):
    """qsa_indexer_prefill_handoff: the prefill call's block keys and trailing raw keys into the pool tails."""
    B, S, di = idxK.shape
    nflat, tpp, Hkv, phd = pool.shape
    if tpp != 128 or tuple(page_table.shape[:2]) != (B, 2):
        raise ValueError("indexer_prefill_handoff: shape mismatch")
    p = QsaIndexerHandoffParams(
        idxK=_ptr(idxK, torch.float16, "idxK"), contextLengths=_ptr(ctx, torch.int32, "contextLengths"),
        workspace=_ptr(workspace, None, "workspace"), workspaceBytes=workspace.numel() * workspace.element_size(),
        kvPool=_ptr(pool, torch.float16, "kvPool"), pageTable=_ptr(page_table, torch.int32, "pageTable"),
        batchSize=B, seqLen=S, headDim=di, compressRatio=ratio, numKVHeads=Hkv, kvHeadDim=D, poolHeadDim=phd,
        numFlatPages=nflat, maxPagesPerSeq=page_table.shape[-1], stream=_stream(stream))
    _check(lib().qsa_indexer_prefill_handoff(ctypes.byref(p)))


def rope_qkv(qkv, wq, wk, ctx, q_out, *, Hq, Hkv, rot, theta, eps, k_out=None, v_out=None, pool=None,
             page_table=None, stream=None):
    """qsa_rope_qkv: packed qkv fp16 [B,S,Hq+2Hkv,D] -> q_out [B,S,Hq,D]; optional dense k_out / v_out
    [B,S,Hkv,D] and pool K/V rows through the page table."""
    B, S, NH, D = qkv.shape
    if NH != Hq + 2 * Hkv or tuple(q_out.shape) != (B, S, Hq, D):
        raise ValueError("rope_qkv: shape mismatch")
    for t in (k_out, v_out):
        if t is not None and tuple(t.shape) != (B, S, Hkv, D):
            raise ValueError("rope_qkv: k_out/v_out shape mismatch")
    nflat = phd = mpp = 0
    if pool is not None:
        nflat, tpp, ph, phd = pool.shape
        if tpp != 128 or ph != Hkv or page_table is None or tuple(page_table.shape[:2]) != (B, 2):
            raise ValueError("rope_qkv: pool/page table shape mismatch")
        mpp = page_table.shape[-1]
    p = QsaRopeQkvParams(
        qkv=_ptr(qkv, torch.float16, "qkv"), qNormW=_ptr(wq, torch.float32, "qNormW"),
        kNormW=_ptr(wk, torch.float32, "kNormW"), contextLengths=_ptr(ctx, torch.int32, "contextLengths"),
        qOut=_ptr(q_out, torch.float16, "q_out"), kOut=_ptr(k_out, torch.float16, "k_out"),
        vOut=_ptr(v_out, torch.float16, "v_out"), kvPool=_ptr(pool, torch.float16, "kvPool"),
        pageTable=_ptr(page_table, torch.int32, "pageTable"), batchSize=B, seqLen=S, numQHeads=Hq,
        numKVHeads=Hkv, headDim=D, rotDim=rot, poolHeadDim=phd, numFlatPages=nflat, maxPagesPerSeq=mpp,
        ropeTheta=theta, rmsNormEps=eps, stream=_stream(stream))
    _check(lib().qsa_rope_qkv(ctypes.byref(p)))


def sparse_prefill(q, k, v, indices, ctx, out, scale, stream=None, status=None, impl="mma"):
    """qsa_sparse_prefill (fp16 tensors) or qsa_sparse_prefill_bf16 (bfloat16 tensors):
    q/out [B,S,Hq,D], k/v [B,S,Hkv,D], indices int32 [B,S,topK]; status: optional int32 device
    tensor whose first word collects the error bits.  impl="tcgen05" calls the tensor-core
    variants qsa_sparse_prefill_tcgen05(_bf16) with the same arguments."""
    if impl not in ("mma", "tcgen05"):
        raise ValueError("sparse_prefill: impl must be 'mma' or 'tcgen05'")
    et = q.dtype
    if et not in (torch.float16, torch.bfloat16):
        raise ValueError("sparse_prefill: q must be float16 or bfloat16")
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    topK = indices.shape[-1]
    if tuple(k.shape) != (B, S, Hkv, D) or tuple(v.shape) != (B, S, Hkv, D) or tuple(out.shape) != (B, S, Hq, D) \
            or indices.numel() != B * S * topK:
        raise ValueError("sparse_prefill: shape mismatch")
    p = QsaSparsePrefillParams(
        qPtr=_ptr(q, et, "q"), kPtr=_ptr(k, et, "k"), vPtr=_ptr(v, et, "v"),
        oPtr=_ptr(out, et, "out"), indices=_ptr(indices, torch.int32, "indices"),
        contextLengths=_ptr(ctx, torch.int32, "contextLengths"), batchSize=B, seqLen=S, numQHeads=Hq,
        numKVHeads=Hkv, headDim=D, topK=topK, attentionScale=scale, stream=_stream(stream),
        status=None if status is None else _ptr(status, torch.int32, "status"))
    name = "qsa_sparse_prefill" + ("_tcgen05" if impl == "tcgen05" else "") + ("_bf16" if et == torch.bfloat16 else "")
    _check(getattr(lib(), name)(ctypes.byref(p)))


def sparse_decode(q, pool, page_table, indices, ctx, out, partial_o, partial_stats, counters, *, D, scale,
                  stream=None, status=None):
    """qsa_sparse_decode (fp16) or qsa_sparse_decode_bf16 (bfloat16 q/pool/out): q/out [B,1,Hq,D]; split-K
    over the pool through the page table."""
    et = q.dtype
    if et not in (torch.float16, torch.bfloat16):
        raise ValueError("sparse_decode: q must be float16 or bfloat16")
    B = q.shape[0]
    Hq = q.shape[-2]
    nflat, tpp, Hkv, phd = pool.shape
    topK = indices.shape[-1]
    if q.numel() != B * Hq * D or out.numel() != B * Hq * D or indices.numel() != B * topK or tpp != 128:
        raise ValueError("sparse_decode: shape mismatch")
    p = QsaSparseDecodeParams(
        qPtr=_ptr(q, et, "q"), kvPoolPtr=_ptr(pool, et, "kvPool"),
        pageTable=_ptr(page_table, torch.int32, "pageTable"), indices=_ptr(indices, torch.int32, "indices"),
        contextLengths=_ptr(ctx, torch.int32, "contextLengths"), oPtr=_ptr(out, et, "out"),
        partialO=_ptr(partial_o, torch.float32, "partialO"),
        partialStats=_ptr(partial_stats, torch.float32, "partialStats"),
        splitCounters=_ptr(counters, torch.int32, "splitCounters"), batchSize=B, numQHeads=Hq, numKVHeads=Hkv,
        headDim=D, poolHeadDim=phd, numFlatPages=nflat, maxPagesPerSeq=page_table.shape[-1], topK=topK,
        attentionScale=scale, stream=_stream(stream),
        status=None if status is None else _ptr(status, torch.int32, "status"))
    fn = lib().qsa_sparse_decode_bf16 if et == torch.bfloat16 else lib().qsa_sparse_decode
    _check(fn(ctypes.byref(p)))


def gather_scratch(B: int, Hkv: int, D: int, topK: int, dtype=torch.float16, device="cuda"):
    """Buffers for gather_selected: (scratch [2*B*P, 128, Hkv, D], page table int32 [B, 2, P],
    indices int32 [B, 1, topK], lengths int32 [B]), P = ceil(topK / 128)."""
    P = int(lib().qsa_gather_scratch_pages(topK))
    n = int(lib().qsa_gather_scratch_elems(B, Hkv, D, topK))
    if P < 1 or n != 2 * B * P * 128 * Hkv * D:
        raise ValueError("gather_scratch: invalid sizes")
    return (torch.empty((2 * B * P, 128, Hkv, D), dtype=dtype, device=device),
            torch.empty((B, 2, P), dtype=torch.int32, device=device),
            torch.empty((B, 1, topK), dtype=torch.int32, device=device),
            torch.empty((B,), dtype=torch.int32, device=device))


def gather_selected(pool, page_table, indices, ctx, scratch, scratch_pt, scratch_idx, scratch_len, *, D,
                    stream=None):
    """qsa_gather_selected: the K/V rows a decode list names, from the pool [numFlat, 128, Hkv, poolHeadDim]
    into contiguous scratch described as a paged pool (see gather_scratch)."""
    et = pool.dtype
    if et not in (torch.float16, torch.bfloat16) or scratch.dtype != et:
        raise ValueError("gather_selected: pool and scratch must share a float16 or bfloat16 dtype")
    nflat, tpp, Hkv, phd = pool.shape
    B, topK = ctx.shape[0], indices.shape[-1]
    P = scratch_pt.shape[-1]
    if tpp != 128 or tuple(page_table.shape[:2]) != (B, 2) or indices.numel() != B * topK \
            or tuple(scratch.shape) != (2 * B * P, 128, Hkv, D) or tuple(scratch_pt.shape) != (B, 2, P) \
            or scratch_idx.numel() != B * topK or scratch_len.numel() != B:
        raise ValueError("gather_selected: shape mismatch")
    p = QsaGatherParams(
        kvPool=_ptr(pool, et, "pool"), pageTable=_ptr(page_table, torch.int32, "pageTable"),
        indices=_ptr(indices, torch.int32, "indices"), contextLengths=_ptr(ctx, torch.int32, "contextLengths"),
        scratch=_ptr(scratch, et, "scratch"), scratchPageTable=_ptr(scratch_pt, torch.int32, "scratchPageTable"),
        scratchIndices=_ptr(scratch_idx, torch.int32, "scratchIndices"),
        scratchLengths=_ptr(scratch_len, torch.int32, "scratchLengths"), batchSize=B, numKVHeads=Hkv, headDim=D,
        poolHeadDim=phd, numFlatPages=nflat, maxPagesPerSeq=page_table.shape[-1], topK=topK,
        stream=_stream(stream))
    _check(lib().qsa_gather_selected(ctypes.byref(p)))


def sparse_decode_noalloc(q, pool, page_table, indices, ctx, out, *, D, scale, stream=None):
    """qsa_sparse_decode_noalloc: sparse_decode with the library's own fixed scratch (no workspace
    arguments; batch * KV heads <= 256).  Concurrent calls on one GPU race on that scratch."""
    B = q.shape[0]
    Hq = q.shape[-2]
    nflat, tpp, Hkv, phd = pool.shape
    topK = indices.shape[-1]
    if q.numel() != B * Hq * D or out.numel() != B * Hq * D or indices.numel() != B * topK or tpp != 128:
        raise ValueError("sparse_decode_noalloc: shape mismatch")
    p = QsaSparseDecodeParams(
        qPtr=_ptr(q, torch.float16, "q"), kvPoolPtr=_ptr(pool, torch.float16, "kvPool"),
        pageTable=_ptr(page_table, torch.int32, "pageTable"), indices=_ptr(indices, torch.int32, "indices"),
        contextLengths=_ptr(ctx, torch.int32, "contextLengths"), oPtr=_ptr(out, torch.float16, "out"),
        partialO=None, partialStats=None, splitCounters=None, batchSize=B, numQHeads=Hq, numKVHeads=Hkv,
        headDim=D, poolHeadDim=phd, numFlatPages=nflat, maxPagesPerSeq=page_table.shape[-1], topK=topK,
        attentionScale=scale, stream=_stream(stream))
    _check(lib().qsa_sparse_decode_noalloc(ctypes.byref(p)))
