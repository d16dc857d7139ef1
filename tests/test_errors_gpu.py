"""Failure handling on the GPU without faulting it: bad indices are caught in
the kernels and reported through the error word; bounded waits give up and
report; host checks reject bad arguments before launching."""
import pytest
import torch

import kvgen
from decode_attention_kv_softmax_b300.kvdec import (DEVERR_BAD_PAGE, DEVERR_SEQLEN,
                                                     DEVERR_TIMEOUT, KvdecError)

pytestmark = pytest.mark.gpu


def test_bad_page_reported_not_faulted(cuda_lib):
    case = kvgen.gqa_case(2, 8, 2, 128, seqlens=[200, 100], paged=True, seed=41, device="cuda")
    case.block_table[0, 1] = case.k.shape[0] + 5        # out of range
    case.block_table[1, 0] = -3
    flag = cuda_lib.new_error_flag()
    out, _ = cuda_lib.gqa_decode(case.q, case.k, case.v, case.seqlens, case.block_table,
                                 error_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() & DEVERR_BAD_PAGE
    assert torch.isfinite(out).all()


def test_seqlen_beyond_capacity_reported(cuda_lib):
    case = kvgen.gqa_case(2, 8, 2, 128, seqlens=[64, 64], cap=64, seed=42, device="cuda")
    case.seqlens[1] = 1000
    flag = cuda_lib.new_error_flag()
    cuda_lib.gqa_decode(case.q, case.k, case.v, case.seqlens, error_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() & DEVERR_SEQLEN


def test_append_bad_position_reported(cuda_lib):
    case = kvgen.mla_case(2, 2, seqlens=[10, 10], seed=43, device="cuda")
    ckv, kr = kvgen.append_inputs_mla(2, seed=44, device="cuda")
    pos = torch.tensor([5, 10 ** 6], dtype=torch.int32, device="cuda")
    flag = cuda_lib.new_error_flag()
    cuda_lib.append_rope_mla(case.cache, case.block_table, pos, ckv, kr, error_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() & DEVERR_SEQLEN


def test_bounded_wait_times_out_cleanly(cuda_lib):
    """A barrier that nothing completes: the wait gives up after ~2 ms,
    reports KVDEC_DEVERR_TIMEOUT, and the context keeps working."""
    flag = cuda_lib.new_error_flag()
    cuda_lib.selftest_wait_timeout(2_000_000, flag)
    torch.cuda.synchronize()
    assert flag.item() == DEVERR_TIMEOUT
    case = kvgen.gqa_case(1, 4, 2, 64, seqlens=[10], seed=45, device="cuda")
    out, _ = cuda_lib.gqa_decode(case.q, case.k, case.v, case.seqlens)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()


def test_host_rejects_bad_arguments(cuda_lib):
    case = kvgen.gqa_case(1, 8, 2, 128, seqlens=[10], seed=46, device="cuda")
    q_mis = torch.empty(8 * 128 + 1, dtype=torch.bfloat16, device="cuda")[1:].view(1, 8, 128)
    with pytest.raises(KvdecError, match="aligned"):
        cuda_lib.gqa_decode(q_mis, case.k, case.v, case.seqlens)
    with pytest.raises(KvdecError, match="workspace"):
        cuda_lib.gqa_decode(case.q, case.k, case.v, case.seqlens,
                            workspace=torch.zeros(16, dtype=torch.uint8, device="cuda"))
    k96 = torch.zeros(1, 2, 16, 96, dtype=torch.bfloat16, device="cuda")
    q96 = torch.zeros(1, 8, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(KvdecError, match="head_dim 96"):
        cuda_lib.gqa_decode(q96, k96, k96, case.seqlens)
    for bad in (-0.5, float("nan"), float("inf")):
        with pytest.raises(KvdecError, match="scale"):
            cuda_lib.gqa_decode(case.q, case.k, case.v, case.seqlens, scale=bad)
    mc = kvgen.mla_case(1, 128, seqlens=[70], seed=47, device="cuda")
    with pytest.raises(KvdecError, match="scale"):
        cuda_lib.mla_decode_absorbed(mc.q_abs, mc.q_rope, mc.cache, mc.block_table, mc.seqlens,
                                     scale=-0.1)
