"""GPU parity of kvdec_mla_decode_absorbed (tcgen05 MLA decode over the paged
576-wide latent cache) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import kvgen
import oracle
from parity import assert_attn_close, assert_lse_close, f64, mla_full_oracle

pytestmark = pytest.mark.gpu


def run(kv, case, **kw):
    """One decode through the C ABI; a valid launch leaves the device error
    word clear (no bad index, no wait that ran out)."""
    flag = kv.new_error_flag()
    out, lse = kv.mla_decode_absorbed(case.q_abs, case.q_rope, case.cache, case.block_table,
                                      case.seqlens, scale=case.scale, error_flag=flag, **kw)
    torch.cuda.synchronize()
    assert flag.item() == 0, f"device error word {flag.item():#x}"
    return out, lse


def full_oracle(case):
    return oracle.mla_decode_absorbed(f64(case.q_abs), f64(case.q_rope), f64(case.cache),
                                      case.block_table.cpu().numpy(), case.seqlens.cpu().numpy(),
                                      case.scale)


@pytest.mark.parametrize("sl", [[100, 700], [1, 64, 65], [64], [3000, 17, 129, 4096]])
def test_small_full_parity(cuda_lib, sl):
    case = kvgen.mla_case(len(sl), 128, seqlens=sl, seed=200 + len(sl), device="cuda")
    out, lse = run(cuda_lib, case)
    ref, lref = full_oracle(case)
    assert_attn_close(out, ref, "mla")
    assert_lse_close(lse, lref, "mla lse")


def test_many_short_sequences(cuda_lib):
    """The largest batch the kernel takes: every thread of the block-wide
    tile scan carries a sequence, and the tile table fills its shared
    memory."""
    g = torch.Generator().manual_seed(5)
    sl = torch.randint(0, 200, (cuda_lib.load().kvdec_mla_max_batch(),), generator=g)
    sl[::37] = 0                         # some sequences are empty
    sl = sl.tolist()
    case = kvgen.mla_case(len(sl), 128, seqlens=sl, seed=217, device="cuda")
    out, lse = run(cuda_lib, case)
    ref, lref = mla_full_oracle(case)
    assert_attn_close(out, ref, "many")
    assert_lse_close(lse, lref)
    empty = [b for b, s in enumerate(sl) if s == 0]
    assert empty and all(torch.all(out[b] == 0) for b in empty)


@pytest.mark.parametrize("max_ctas", [8, 0])
def test_work_items_without_pages(cuda_lib, max_ctas):
    """The split schedule charges every sequence start (empty ones too) a
    few pages, so with hundreds of empty sequences and one long one the cut
    points can fall where no page lies: some CTA pairs get no pages, the
    long sequence's pieces sit in consecutive work items, and the empty
    sequences are still written (0 and lse = -inf)."""
    sl = [0] * 300
    sl[250] = 5000      # with the full grid: cut into two pieces, most items empty
    sl[17] = 5
    case = kvgen.mla_case(len(sl), 128, seqlens=sl, seed=219, device="cuda")
    out, lse = run(cuda_lib, case, max_ctas=max_ctas)
    ref, lref = mla_full_oracle(case)
    assert_attn_close(out, ref, f"sparse max_ctas={max_ctas}")
    assert_lse_close(lse, lref)
    empty = [b for b, s in enumerate(sl) if s == 0]
    assert all(torch.all(out[b] == 0) for b in empty)
    assert torch.isneginf(lse[empty]).all()


@pytest.mark.parametrize("max_ctas", [2, 4, 6, 14, 0])
def test_split_invariance(cuda_lib, max_ctas):
    """Sequences cut across CTA pairs merge to the same result."""
    case = kvgen.mla_case(3, 128, seqlens=[2500, 640, 5], seed=211, device="cuda")
    ref, lref = full_oracle(case)
    out, lse = run(cuda_lib, case, max_ctas=max_ctas)
    assert_attn_close(out, ref, f"max_ctas={max_ctas}")
    assert_lse_close(lse, lref)


def test_empty_sequences_and_bf16(cuda_lib):
    case = kvgen.mla_case(3, 128, seqlens=[0, 300, 0], seed=212, device="cuda")
    out, lse = run(cuda_lib, case, out_dtype=torch.bfloat16)
    assert out.dtype == torch.bfloat16
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    assert torch.isneginf(lse[0]).all() and torch.isneginf(lse[2]).all()
    ref, lref = full_oracle(case)
    assert_attn_close(out, ref, "bf16")
    assert_lse_close(lse, lref)


def test_default_scale_is_192(cuda_lib):
    """scale 0 selects 1/sqrt(128 + 64) ([ARG] §四.5)."""
    case = kvgen.mla_case(1, 128, seqlens=[333], seed=213, device="cuda")
    out, _ = cuda_lib.mla_decode_absorbed(case.q_abs, case.q_rope, case.cache, case.block_table,
                                          case.seqlens)
    torch.cuda.synchronize()
    ref, _ = full_oracle(case)
    assert_attn_close(out, ref)


def test_shared_pages(cuda_lib):
    case = kvgen.mla_case(2, 128, seqlens=[700, 700], seed=214, device="cuda")
    case.block_table[1] = case.block_table[0]
    case.q_abs[1] = case.q_abs[0]
    case.q_rope[1] = case.q_rope[0]
    out, _ = run(cuda_lib, case)
    assert_attn_close(out[0], f64(out[1]), "aliased pages", atol=5e-3, row_rtol=5e-3)
    ref, _ = full_oracle(case)
    assert_attn_close(out, ref)


def test_rope_part_is_used(cuda_lib):
    """Zeroing q_rope changes the result exactly as the oracle says: the
    decoupled rope term of the score is not dropped."""
    case = kvgen.mla_case(2, 128, seqlens=[400, 90], seed=215, device="cuda")
    case.q_rope.mul_(8.0)
    out, _ = run(cuda_lib, case)
    ref, _ = full_oracle(case)
    assert_attn_close(out, ref, "scaled rope")
    case.q_rope.zero_()
    out0, _ = run(cuda_lib, case)
    ref0, _ = full_oracle(case)
    assert_attn_close(out0, ref0, "no rope")
    assert np.abs(ref - ref0).max() > 0.05


@pytest.mark.parametrize("name", ["C3", "C4-MLA"])
def test_full_size_full_output(cuda_lib, name):
    """The named workloads at full size, in the launch configuration the
    benchmark uses: every (b, h) row of the latent output and of lse against
    the oracle."""
    case = kvgen.config_case(name, device="cuda")
    out, lse = run(cuda_lib, case)
    ref, lref = mla_full_oracle(case)
    assert_attn_close(out, ref, name)
    assert_lse_close(lse, lref, name)


def test_bad_page_reported(cuda_lib):
    case = kvgen.mla_case(2, 128, seqlens=[200, 100], seed=216, device="cuda")
    case.block_table[0, 1] = case.cache.shape[0] + 3
    flag = cuda_lib.new_error_flag()
    out, _ = cuda_lib.mla_decode_absorbed(case.q_abs, case.q_rope, case.cache, case.block_table,
                                          case.seqlens, error_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() & cuda_lib.DEVERR_BAD_PAGE
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("max_ctas", [2, 0])
def test_lazy_rescale_heavy_tail(cuda_lib, max_ctas):
    """Heavy-tailed rope scores (logits up to ~20): row maxima jump by more
    than 2^8 at random pages of both parities, so O is rescaled mid-sequence
    by both softmax groups; one pair (max_ctas=2) walks every page."""
    case = kvgen.mla_case(2, 128, seqlens=[3000, 1100], seed=218, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(9)
    case.q_rope.zero_()
    case.q_rope[:, :, 0] = (1.5 * torch.randn((2, 128), generator=g, device="cuda")).to(torch.bfloat16)
    spikes = torch.empty(case.cache.shape[:2], device="cuda").exponential_(1.0, generator=g)
    case.cache[:, :, 512] = (12.0 * spikes).to(torch.bfloat16)
    out, lse = run(cuda_lib, case, max_ctas=max_ctas)
    ref, lref = full_oracle(case)
    # the rope part of the scores alone already moves some row maxima by
    # more than 8 (log2 units) after the first page
    t = torch.arange(3000)
    k0 = case.cache.cpu().double()[case.block_table.cpu()[0, t // 64].long(), t % 64, 512]
    sc = case.q_rope.cpu().double()[0, :, :1] * k0[None, :] * case.scale / np.log(2)
    assert ((sc.max(1).values - sc[:, :64].max(1).values) > 8.0).any()
    assert_attn_close(out, ref, f"heavy tail, max_ctas={max_ctas}")
    assert_lse_close(lse, lref)
