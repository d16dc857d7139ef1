"""GPU parity of kvdec_combine_splits and kvdec_append_rope against the
oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import kvgen
import oracle
from parity import assert_attn_close, assert_lse_close, f64

pytestmark = pytest.mark.gpu


def bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("S,R,D", [(1, 5, 128), (4, 33, 512), (7, 10, 100), (64, 3, 64)])
def test_combine_matches_oracle(cuda_lib, S, R, D):
    g = torch.Generator().manual_seed(S * 1000 + D)
    po = torch.randn(S, R, D, generator=g)
    plse = torch.randn(S, R, generator=g) * 3
    plse[0, 0] = -float("inf")            # an empty piece
    counts = torch.randint(0, S + 1, (R,), generator=g, dtype=torch.int32)
    counts[0] = S
    out_init = torch.full((R, D), 7.0)
    out = out_init.cuda()
    got, lse = cuda_lib.combine_splits(po.cuda(), plse.cuda(), counts.cuda(), out=out)
    torch.cuda.synchronize()
    ref, lref = oracle.combine_splits(po.double().numpy(), plse.double().numpy(), counts.numpy())
    c = counts.numpy()
    used = c > 0
    assert_attn_close(got.cpu()[used], ref[used], "combine")
    assert_lse_close(lse.cpu()[used], lref[used])
    assert torch.all(got.cpu()[~torch.as_tensor(used)] == 7.0)   # untouched rows


def test_combine_all_empty_row(cuda_lib):
    po = torch.randn(3, 2, 16).cuda()
    plse = torch.full((3, 2), -float("inf")).cuda()
    plse[1, 1] = 0.5
    out, lse = cuda_lib.combine_splits(po, plse)
    torch.cuda.synchronize()
    assert torch.all(out[0] == 0) and torch.isneginf(lse[0])
    assert torch.allclose(out[1], po[1, 1], atol=1e-6) and abs(lse[1].item() - 0.5) < 1e-6


def test_combine_bf16_out(cuda_lib):
    po = torch.randn(5, 9, 128).cuda()
    plse = torch.randn(5, 9).cuda()
    out, _ = cuda_lib.combine_splits(po, plse, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    ref, _ = oracle.combine_splits(po.double().cpu().numpy(), plse.double().cpu().numpy())
    assert_attn_close(out, ref)


def test_split_then_combine_equals_unsplit(cuda_lib):
    """Decode pieces of one sequence separately (the sequence cut at token
    boundaries), merge them with kvdec_combine_splits: equals the unsplit
    decode ([ARG] §五.2)."""
    case = kvgen.gqa_case(1, 8, 2, 128, seqlens=[1000], cap=1024, seed=21, device="cuda")
    bounds = [0, 128, 640, 1000]
    parts, plses = [], []
    for a, e in zip(bounds[:-1], bounds[1:]):
        k = case.k[:, :, a:e].contiguous()
        v = case.v[:, :, a:e].contiguous()
        o, l = cuda_lib.gqa_decode(case.q, k, v, torch.tensor([e - a], dtype=torch.int32, device="cuda"),
                                   scale=case.scale)
        parts.append(o.reshape(8, 128))
        plses.append(l.reshape(8))
    out, lse = cuda_lib.combine_splits(torch.stack(parts), torch.stack(plses))
    full, lfull = cuda_lib.gqa_decode(case.q, case.k, case.v, case.seqlens, scale=case.scale)
    torch.cuda.synchronize()
    assert_attn_close(out, f64(full.reshape(8, 128)), atol=2e-3, row_rtol=2e-3)
    assert_lse_close(lse, f64(lfull.reshape(8)), atol=1e-3)


def test_append_mla(cuda_lib):
    sl_new = [1, 64, 65, 201, 131072]
    case = kvgen.mla_case(5, 2, seqlens=sl_new, seed=31, device="cuda", spare_pages=3)
    pos = torch.tensor([s - 1 for s in sl_new], dtype=torch.int32, device="cuda")
    before = bits(case.cache)
    ckv, kr = kvgen.append_inputs_mla(5, seed=32, device="cuda")
    flag = cuda_lib.new_error_flag()
    cuda_lib.append_rope_mla(case.cache, case.block_table, pos, ckv, kr, error_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    after = bits(case.cache)
    ref = oracle.append_rope_mla(before, case.block_table.cpu().numpy(), pos.cpu().numpy(),
                                 bits(ckv), bits(kr))
    # every byte outside the new rows untouched, c_kv bit-exact
    bt = case.block_table.cpu().numpy()
    mask = np.ones(before.shape[:2], bool)
    for b, p in enumerate(pos.cpu().numpy()):
        mask[bt[b, p // 64], p % 64] = False
    assert np.array_equal(after[mask], before[mask])
    assert np.array_equal(after[..., :512], ref[..., :512])
    # rotated rope key within one bf16 ulp of the fp64 oracle
    d = np.abs(after[..., 512:].astype(np.int32) - ref[..., 512:].astype(np.int32))
    assert d.max() <= 1


@pytest.mark.parametrize("paged", [False, True])
def test_append_gqa(cuda_lib, paged):
    B, n_kv, d = 4, 8, 128
    sl_new = [1, 64, 300, 4096]
    case = kvgen.gqa_case(B, 8 * n_kv, n_kv, d, seqlens=sl_new, cap=4096, paged=paged,
                          seed=33, device="cuda")
    pos = torch.tensor([s - 1 for s in sl_new], dtype=torch.int32, device="cuda")
    kb, vb = bits(case.k), bits(case.v)
    k_new, v_new = kvgen.append_inputs_gqa(B, n_kv, d, seed=34, device="cuda")
    cuda_lib.append_rope_gqa(case.k, case.v, pos, k_new, v_new, case.block_table)
    torch.cuda.synchronize()
    bt = None if case.block_table is None else case.block_table.cpu().numpy()
    rk, rv = oracle.append_rope_gqa(kb, vb, pos.cpu().numpy(), bits(k_new), bits(v_new), bt)
    assert np.array_equal(bits(case.v), rv)
    dk = np.abs(bits(case.k).astype(np.int32) - rk.astype(np.int32))
    assert dk.max() <= 1
    assert (dk > 0).sum() <= 4    # rare round-to-nearest ties only


def test_append_then_decode_sees_new_token(cuda_lib):
    """A decode step: append the new token at slot len, then attend over
    len + 1 tokens; the result matches the oracle on the appended cache."""
    case = kvgen.gqa_case(2, 8, 2, 128, seqlens=[99, 64], cap=128, seed=35, device="cuda")
    k_new, v_new = kvgen.append_inputs_gqa(2, 2, 128, seed=36, device="cuda")
    cuda_lib.append_rope_gqa(case.k, case.v, case.seqlens, k_new, v_new)
    sl1 = case.seqlens + 1
    out, _ = cuda_lib.gqa_decode(case.q, case.k, case.v, sl1, scale=case.scale)
    torch.cuda.synchronize()
    ref, _ = oracle.gqa_decode(f64(case.q), f64(case.k), f64(case.v), sl1.cpu().numpy(), case.scale)
    assert_attn_close(out, ref)
