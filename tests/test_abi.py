"""The C-ABI library without a GPU: it loads, exports every symbol that
include/qsa.h declares, its params structs match the C layout, and its
host-only paths (sizes, constants, parameter validation) behave.  No call here
reaches a kernel launch."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "qsa.h")


@pytest.fixture(scope="module")
def binding():
    from block_sparse_gqa_qsa_gb300 import build, _binding
    build.build()
    _binding.lib()
    return _binding


def declared_functions():
    src = open(HEADER).read()
    return re.findall(r"^QSA_API\s+[\w\s\*]+?\b(qsa_\w+)\s*\(", src, flags=re.M)


def test_every_declared_symbol_is_exported(binding):
    names = declared_functions()
    assert len(names) >= 16
    L = binding.lib()
    for n in names:
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (qsa_\w+)", out))
    assert exported == set(names)


def test_struct_layouts_match_c(binding, tmp_path):
    structs = {"QsaIndexerPrefillParams": binding.QsaIndexerPrefillParams,
               "QsaIndexerDecodeParams": binding.QsaIndexerDecodeParams,
               "QsaSparsePrefillParams": binding.QsaSparsePrefillParams,
               "QsaSparseDecodeParams": binding.QsaSparseDecodeParams,
               "QsaIndexerHandoffParams": binding.QsaIndexerHandoffParams,
               "QsaRopeQkvParams": binding.QsaRopeQkvParams,
               "QsaGatherParams": binding.QsaGatherParams}
    lines = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{HEADER}"', "int main(void) {"]
    for s, cls in structs.items():
        lines.append(f'printf("{s} size %zu\\n", sizeof({s}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("{s} {f} %zu\\n", offsetof({s}, {f}));')
    lines.append("return 0; }")
    c = tmp_path / "layout.c"
    c.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", str(c), "-o", str(exe)], check=True)
    got = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    for line in filter(None, got):
        s, f, v = line.split()
        cls = structs[s]
        want = ctypes.sizeof(cls) if f == "size" else getattr(cls, f).offset
        assert int(v) == want, line


def test_constants_and_sizes(binding):
    L = binding.lib()
    assert L.qsa_sparse_decode_max_splits() == 8
    assert L.qsa_sparse_decode_partial_rows() == 16
    assert L.qsa_indexer_prefill_max_seq_len() == 1 << 24
    assert L.qsa_indexer_prefill_max_blocks() == 1 << 24
    B, Hkv, D = 3, 4, 128
    po, ps, pc = binding.sparse_decode_workspace_elems(B, Hkv, D)
    assert (po, ps, pc) == (B * Hkv * 8 * 16 * D, B * Hkv * 8 * 2 * 16, B * Hkv)
    # status, block keys (256-byte rounded), work counter, 320 score slots of 8 rows x S/r floats
    kb = -(-(2 * 250 * 128 * 2) // 256) * 256
    assert binding.indexer_prefill_workspace_size(2, 1000, 128, 4) == 256 + kb + 256 + 320 * 8 * 250 * 4
    # linear in S: doubling S doubles every term that depends on it
    w1 = binding.indexer_prefill_workspace_size(1, 65536, 128, 4) - 512
    w2 = binding.indexer_prefill_workspace_size(1, 131072, 128, 4) - 512
    assert w2 == 2 * w1
    assert binding.indexer_prefill_workspace_size(0, 1000, 128, 4) == 0
    # scores, tie keys and tie ids: 12 bytes per possible block of every sequence, at least
    assert binding.indexer_decode_workspace_size(8, 4096, 4, 512) >= 8 * 4096 * 32 * 12
    assert binding.indexer_decode_workspace_size(8, 4096, 3, 512) == 0  # 3 does not divide a page
    assert L.qsa_sparse_prefill_can_implement(32, 4, 128) == 1
    assert L.qsa_sparse_prefill_can_implement(64, 2, 128) == 0  # group 32 > 16
    assert L.qsa_sparse_prefill_can_implement(32, 4, 64) == 0
    assert L.qsa_sparse_decode_can_implement(64, 8, 128, 256) == 1
    assert L.qsa_gather_scratch_pages(2051) == 17 and L.qsa_gather_scratch_pages(128) == 1
    assert L.qsa_gather_scratch_elems(3, 4, 128, 2051) == 2 * 3 * 17 * 128 * 4 * 128
    assert L.qsa_gather_scratch_elems(0, 4, 128, 2051) == 0
    assert L.qsa_sparse_decode_can_implement(64, 8, 128, 100) == 0
    assert L.qsa_status_string(2) == b"QSA_ERR_UNSUPPORTED"
    out = ctypes.c_int32(0)
    assert L.qsa_last_device_error(None, None, ctypes.byref(out)) == binding.QSA_ERR_INVALID_ARG
    assert L.qsa_last_device_error(ctypes.c_void_p(1 << 20), None, None) == binding.QSA_ERR_INVALID_ARG


def _call(binding, fn, params):
    return getattr(binding.lib(), fn)(ctypes.byref(params) if params is not None else None)


def test_validation_rejects_before_launch(binding):
    L = binding.lib()
    for fn in ("qsa_indexer_prefill", "qsa_indexer_decode", "qsa_sparse_prefill", "qsa_sparse_decode",
               "qsa_indexer_prefill_handoff", "qsa_rope_qkv", "qsa_sparse_prefill_bf16", "qsa_sparse_decode_bf16",
               "qsa_sparse_prefill_tcgen05", "qsa_sparse_prefill_tcgen05_bf16",
               "qsa_gather_selected"):
        assert getattr(L, fn)(None) == binding.QSA_ERR_INVALID_ARG
    fake = 1 << 20  # never dereferenced: every case below fails validation first
    sp = binding.QsaSparsePrefillParams(qPtr=fake, kPtr=fake, vPtr=fake, oPtr=fake, indices=fake,
                                        contextLengths=fake, batchSize=1, seqLen=16, numQHeads=32, numKVHeads=4,
                                        headDim=128, topK=67, attentionScale=0.1)
    sp.numQHeads = 30
    assert _call(binding, "qsa_sparse_prefill", sp) == binding.QSA_ERR_INVALID_ARG
    assert b"numKVHeads" in L.qsa_last_error_message()
    sp.numQHeads, sp.numKVHeads = 64, 2
    assert _call(binding, "qsa_sparse_prefill", sp) == binding.QSA_ERR_UNSUPPORTED
    sp.numKVHeads, sp.headDim = 4, 64
    assert _call(binding, "qsa_sparse_prefill", sp) == binding.QSA_ERR_UNSUPPORTED
    sp.headDim, sp.vPtr = 128, None
    assert _call(binding, "qsa_sparse_prefill", sp) == binding.QSA_ERR_INVALID_ARG
    sp.vPtr, sp.qPtr = fake, fake + 2
    assert _call(binding, "qsa_sparse_prefill", sp) == binding.QSA_ERR_INVALID_ARG  # misaligned

    ip = binding.QsaIndexerPrefillParams(idxQ=fake, idxK=fake, qNormW=fake, kNormW=fake, contextLengths=fake,
                                         indices=fake, workspace=fake, workspaceBytes=16, batchSize=1,
                                         seqLen=8192, numHeads=8, headDim=128, rotDim=64, compressRatio=4,
                                         budget=512, topK=2050, ropeTheta=1e4, rmsNormEps=1e-6)
    assert _call(binding, "qsa_indexer_prefill", ip) == binding.QSA_ERR_INVALID_ARG  # topK < 2051
    ip.topK = 2051
    assert _call(binding, "qsa_indexer_prefill", ip) == binding.QSA_ERR_WORKSPACE  # 16 bytes
    ip.seqLen = 131072  # long sequences are taken: only the workspace is short
    assert _call(binding, "qsa_indexer_prefill", ip) == binding.QSA_ERR_WORKSPACE
    ip.seqLen = (1 << 24) + 8
    assert _call(binding, "qsa_indexer_prefill", ip) == binding.QSA_ERR_UNSUPPORTED  # past 2^24 rows
    ip.seqLen, ip.batchSize = 1 << 20, 4096
    assert _call(binding, "qsa_indexer_prefill", ip) == binding.QSA_ERR_UNSUPPORTED  # B*S >= 2^31
    ip.batchSize = 1
    ip.seqLen, ip.headDim = 8192, 96
    assert _call(binding, "qsa_indexer_prefill", ip) == binding.QSA_ERR_UNSUPPORTED
    ip.headDim, ip.rotDim = 128, 63
    assert _call(binding, "qsa_indexer_prefill", ip) == binding.QSA_ERR_INVALID_ARG
    ip.rotDim, ip.numHeads = 64, 9
    assert _call(binding, "qsa_indexer_prefill", ip) == binding.QSA_ERR_UNSUPPORTED

    dp = binding.QsaIndexerDecodeParams(idxQ=fake, idxK=fake, qNormW=fake, kNormW=fake, kvPool=fake,
                                        pageTable=fake, contextLengths=fake, indices=fake, workspace=fake,
                                        workspaceBytes=16, batchSize=8, numKVHeads=8, kvHeadDim=128,
                                        poolHeadDim=200, numFlatPages=10, maxPagesPerSeq=4096, numHeads=8,
                                        headDim=128, rotDim=64, compressRatio=4, budget=512, topK=2051,
                                        ropeTheta=1e4, rmsNormEps=1e-6)
    assert _call(binding, "qsa_indexer_decode", dp) == binding.QSA_ERR_INVALID_ARG  # 200 < 128 + 128
    dp.poolHeadDim = 256
    assert _call(binding, "qsa_indexer_decode", dp) == binding.QSA_ERR_WORKSPACE
    dp.compressRatio, dp.topK = 3, 2051
    assert _call(binding, "qsa_indexer_decode", dp) == binding.QSA_ERR_INVALID_ARG
    dp.compressRatio, dp.topK = 2, 1025  # a page's 64 key tails exceed one ring stage
    assert _call(binding, "qsa_indexer_decode", dp) == binding.QSA_ERR_UNSUPPORTED
    dp.compressRatio, dp.topK, dp.batchSize = 4, 2051, 5000
    assert _call(binding, "qsa_indexer_decode", dp) == binding.QSA_ERR_UNSUPPORTED

    hp = binding.QsaIndexerHandoffParams(idxK=fake, contextLengths=fake, workspace=fake, workspaceBytes=16,
                                         kvPool=fake, pageTable=fake, batchSize=2, seqLen=1000, headDim=128,
                                         compressRatio=4, numKVHeads=2, kvHeadDim=128, poolHeadDim=256, numFlatPages=8,
                                         maxPagesPerSeq=8)
    assert _call(binding, "qsa_indexer_prefill_handoff", hp) == binding.QSA_ERR_WORKSPACE  # 16 bytes
    hp.maxPagesPerSeq = 7  # 896 tokens < seqLen
    assert _call(binding, "qsa_indexer_prefill_handoff", hp) == binding.QSA_ERR_INVALID_ARG
    hp.maxPagesPerSeq, hp.headDim = 8, 96
    assert _call(binding, "qsa_indexer_prefill_handoff", hp) == binding.QSA_ERR_UNSUPPORTED
    hp.headDim, hp.poolHeadDim = 128, 200
    assert _call(binding, "qsa_indexer_prefill_handoff", hp) == binding.QSA_ERR_INVALID_ARG
    assert L.qsa_indexer_prefill_handoff(None) == binding.QSA_ERR_INVALID_ARG

    rp = binding.QsaRopeQkvParams(qkv=fake, qNormW=fake, kNormW=fake, contextLengths=fake, qOut=fake, batchSize=1,
                                  seqLen=16, numQHeads=8, numKVHeads=2, headDim=96, rotDim=32, ropeTheta=1e4,
                                  rmsNormEps=1e-6)
    assert _call(binding, "qsa_rope_qkv", rp) == binding.QSA_ERR_UNSUPPORTED  # headDim 96
    rp.headDim, rp.rotDim = 128, 33
    assert _call(binding, "qsa_rope_qkv", rp) == binding.QSA_ERR_INVALID_ARG  # odd rotDim
    rp.rotDim = 24
    assert _call(binding, "qsa_rope_qkv", rp) == binding.QSA_ERR_UNSUPPORTED  # rotDim not a multiple of 16
    rp.rotDim, rp.numQHeads = 64, 300
    assert _call(binding, "qsa_rope_qkv", rp) == binding.QSA_ERR_UNSUPPORTED  # 304 heads * 256 B > 64 KiB row
    rp.numQHeads, rp.qkv = 8, fake + 2
    assert _call(binding, "qsa_rope_qkv", rp) == binding.QSA_ERR_UNSUPPORTED  # qkv not 16-byte aligned
    rp.qkv, rp.kvPool = fake, fake
    assert _call(binding, "qsa_rope_qkv", rp) == binding.QSA_ERR_INVALID_ARG  # pool without a page table
    rp.pageTable, rp.poolHeadDim, rp.numFlatPages, rp.maxPagesPerSeq = fake, 132, 4, 2
    assert _call(binding, "qsa_rope_qkv", rp) == binding.QSA_ERR_UNSUPPORTED  # poolHeadDim not a multiple of 8
    rp.kvPool, rp.qOut = None, None
    assert _call(binding, "qsa_rope_qkv", rp) == binding.QSA_ERR_INVALID_ARG

    gp = binding.QsaGatherParams(kvPool=fake, pageTable=fake, indices=fake, contextLengths=fake, scratch=fake,
                                 scratchPageTable=fake, scratchIndices=fake, scratchLengths=None, batchSize=2,
                                 numKVHeads=4, headDim=128, poolHeadDim=256, numFlatPages=8, maxPagesPerSeq=4,
                                 topK=2051)
    assert _call(binding, "qsa_gather_selected", gp) == binding.QSA_ERR_INVALID_ARG  # no scratchLengths
    gp.scratchLengths, gp.poolHeadDim = fake, 100
    assert _call(binding, "qsa_gather_selected", gp) == binding.QSA_ERR_INVALID_ARG  # poolHeadDim < headDim
    gp.poolHeadDim, gp.numKVHeads = 256, 16
    assert _call(binding, "qsa_gather_selected", gp) == binding.QSA_ERR_UNSUPPORTED  # 16 x 128 > 1024 per row
    gp.numKVHeads, gp.scratch = 4, fake + 8
    assert _call(binding, "qsa_gather_selected", gp) == binding.QSA_ERR_UNSUPPORTED  # scratch not 16-byte aligned
    gp.scratch, gp.topK = fake, 0
    assert _call(binding, "qsa_gather_selected", gp) == binding.QSA_ERR_INVALID_ARG

    sd = binding.QsaSparseDecodeParams(qPtr=fake, kvPoolPtr=fake, pageTable=fake, indices=fake,
                                       contextLengths=fake, oPtr=fake, partialO=None, partialStats=fake,
                                       splitCounters=fake, batchSize=8, numQHeads=64, numKVHeads=8, headDim=128,
                                       poolHeadDim=256, numFlatPages=10, maxPagesPerSeq=4096, topK=2051,
                                       attentionScale=0.1)
    assert _call(binding, "qsa_sparse_decode", sd) == binding.QSA_ERR_WORKSPACE
    sd.partialO, sd.poolHeadDim = fake, 100
    assert _call(binding, "qsa_sparse_decode", sd) == binding.QSA_ERR_INVALID_ARG
    sd.poolHeadDim, sd.numQHeads = 256, 60
    assert _call(binding, "qsa_sparse_decode", sd) == binding.QSA_ERR_INVALID_ARG  # 60 % 8 != 0
    sd.numQHeads, sd.numKVHeads = 64, 2
    assert _call(binding, "qsa_sparse_decode", sd) == binding.QSA_ERR_UNSUPPORTED  # a GQA group of 32
    sd.numKVHeads, sd.topK = 8, 16385
    assert _call(binding, "qsa_sparse_decode", sd) == binding.QSA_ERR_UNSUPPORTED  # the list of a slice on chip
    sd.topK, sd.qPtr = 2051, fake + 4
    assert _call(binding, "qsa_sparse_decode", sd) == binding.QSA_ERR_INVALID_ARG  # q not 16-byte aligned
    sd.qPtr, sd.indices = fake, None
    assert _call(binding, "qsa_sparse_decode_bf16", sd) == binding.QSA_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(binding):
    import torch
    x = torch.zeros(1, 4, 2, 128, dtype=torch.float16)
    k = torch.zeros(1, 4, 1, 128, dtype=torch.float16)
    with pytest.raises(ValueError):
        binding.sparse_prefill(x, k, k, torch.zeros(1, 4, 3, dtype=torch.int32),
                               torch.ones(1, dtype=torch.int32), x.clone(), 0.1)
