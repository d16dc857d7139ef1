"""GPU parity of kvdec_gqa_decode (MHA / GQA / MQA, contiguous and paged)
against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import kvgen
import oracle
from parity import assert_attn_close, assert_lse_close, f64, gqa_full_oracle

pytestmark = pytest.mark.gpu


def run(kv, case, **kw):
    """One decode through the C ABI; a valid launch leaves the device error
    word clear (no bad index, no wait that ran out)."""
    flag = kv.new_error_flag()
    out, lse = kv.gqa_decode(case.q, case.k, case.v, case.seqlens, case.block_table,
                             scale=case.scale, error_flag=flag, **kw)
    torch.cuda.synchronize()
    assert flag.item() == 0, f"device error word {flag.item():#x}"
    return out, lse


def full_oracle(case):
    bt = None if case.block_table is None else case.block_table.cpu().numpy()
    return oracle.gqa_decode(f64(case.q), f64(case.k), f64(case.v),
                             case.seqlens.cpu().numpy(), case.scale, bt)


SMALL = [
    # B, h, n_kv, d, seqlens, paged
    (1, 4, 2, 64, [128], False),                       # the tiny workload's shape
    (3, 8, 2, 128, [1, 65, 4000], False),
    (6, 32, 8, 128, [1, 63, 64, 65, 129, 1000], False),
    (4, 16, 16, 128, [70, 300, 64, 5], False),          # MHA
    (3, 32, 1, 128, [33, 700, 1500], False),            # MQA g = 32, few units: chunks of 16
    (2, 48, 1, 128, [100, 260], False),                 # g = 48: three head chunks of 16
    (160, 32, 1, 128, [1 + (37 * i) % 300 for i in range(160)], False),  # 160 units: 32-row chunks
    (150, 48, 1, 64, [1 + (53 * i) % 200 for i in range(150)], True),    # 32 + 16 rows, d = 64
    (2, 64, 1, 64, [90, 17], False),                    # g = 64, d = 64
    (5, 8, 4, 64, [1, 2, 64, 127, 300], True),
    (3, 64, 8, 128, [5000, 70, 1], True),               # 70B-shaped, paged
    (2, 16, 1, 128, [129, 2000], True),
]


@pytest.mark.parametrize("B,h,n_kv,d,sl,paged", SMALL)
def test_small_full_parity(cuda_lib, B, h, n_kv, d, sl, paged):
    case = kvgen.gqa_case(B, h, n_kv, d, seqlens=sl, paged=paged, seed=100 + B * h + d,
                          device="cuda")
    out, lse = run(cuda_lib, case)
    ref, lref = full_oracle(case)
    assert_attn_close(out, ref, "out")
    assert_lse_close(lse, lref, "lse")


def test_many_short_sequences(cuda_lib):
    """Hundreds of sequences: every thread of the block-wide tile scan
    carries a sequence."""
    g = torch.Generator().manual_seed(6)
    sl = torch.randint(0, 300, (900,), generator=g).tolist()
    case = kvgen.gqa_case(len(sl), 8, 2, 64, seqlens=sl, paged=True, seed=121, device="cuda")
    out, lse = run(cuda_lib, case)
    ref, lref = gqa_full_oracle(case)
    assert_attn_close(out, ref, "many")
    assert_lse_close(lse, lref)


def test_tiny_config(cuda_lib):
    case = kvgen.config_case("C0", device="cuda")
    out, lse = run(cuda_lib, case)
    assert out.dtype == torch.float32 and out.shape == (1, 4, 64)
    ref, lref = full_oracle(case)
    assert_attn_close(out, ref, "C0")
    assert_lse_close(lse, lref)


@pytest.mark.parametrize("max_ctas", [1, 2, 3, 17, 40, 0])
def test_split_invariance(cuda_lib, max_ctas):
    """Any cut of the sequences across CTAs merges to the same result."""
    case = kvgen.gqa_case(4, 16, 4, 128, seqlens=[3000, 64, 1, 700], seed=7, device="cuda")
    ref, lref = full_oracle(case)
    out, lse = run(cuda_lib, case, max_ctas=max_ctas)
    assert_attn_close(out, ref, f"max_ctas={max_ctas}")
    assert_lse_close(lse, lref)


def test_empty_and_full_sequences(cuda_lib):
    case = kvgen.gqa_case(4, 8, 2, 128, seqlens=[0, 256, 0, 1], cap=256, seed=8, device="cuda")
    out, lse = run(cuda_lib, case)
    o = out.cpu().numpy()
    assert np.all(o[0] == 0) and np.all(o[2] == 0)
    assert torch.isneginf(lse[0]).all() and torch.isneginf(lse[2]).all()
    ref, lref = full_oracle(case)
    assert_attn_close(out, ref)
    assert_lse_close(lse, lref)


def test_bf16_output(cuda_lib):
    case = kvgen.gqa_case(3, 32, 8, 128, seqlens=[500, 1, 2100], seed=9, device="cuda")
    out, _ = run(cuda_lib, case, out_dtype=torch.bfloat16)
    assert out.dtype == torch.bfloat16
    ref, _ = full_oracle(case)
    assert_attn_close(out, ref, "bf16 out")


def test_head_axis_mapping(cuda_lib):
    """[CH7] §7.3: query head h must read KV head h // g.  Each KV head holds
    a distinct constant value, so the output names the head it read."""
    B, h, n_kv, d = 2, 12, 3, 128
    case = kvgen.gqa_case(B, h, n_kv, d, seqlens=[200, 77], seed=10, device="cuda")
    for kv in range(n_kv):
        case.v[:, kv] = float(kv + 1)
    out, _ = run(cuda_lib, case)
    want = torch.tensor([hh // (h // n_kv) + 1 for hh in range(h)], dtype=torch.float32)
    assert torch.allclose(out[:, :, 0].cpu(), want.expand(B, h), atol=1e-3)


def test_shared_pages(cuda_lib):
    """Prefix sharing ([ARG] §六.2): two sequences pointing at the same pages
    and with the same query give the same output."""
    case = kvgen.gqa_case(2, 8, 2, 128, seqlens=[300, 300], paged=True, seed=11, device="cuda")
    case.block_table[1] = case.block_table[0]
    case.q[1] = case.q[0]
    out, _ = run(cuda_lib, case)
    # the two rows may be cut at different points across CTAs (so rounded
    # differently), but read the same tokens
    assert_attn_close(out[0], f64(out[1]), "aliased pages", atol=5e-3, row_rtol=5e-3)
    ref, _ = full_oracle(case)
    assert_attn_close(out, ref)


def test_mqa_equals_repeated_mha(cuda_lib):
    """Same q against MQA K/V and against those K/V repeated 32 times along
    the head axis ([KVC-LLM] §四 difference 3): equal outputs."""
    case = kvgen.gqa_case(4, 32, 1, 128, seqlens=[4096] * 4, cap=4096, seed=12, device="cuda")
    out1, _ = run(cuda_lib, case)
    k_rep = case.k.repeat_interleave(32, dim=1).contiguous()
    v_rep = case.v.repeat_interleave(32, dim=1).contiguous()
    out2, _ = cuda_lib.gqa_decode(case.q, k_rep, v_rep, case.seqlens, scale=case.scale)
    torch.cuda.synchronize()
    assert_attn_close(out1, f64(out2), "MQA vs repeated MHA")


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_launch_returns_promptly(cuda_lib, kv_dtype):
    """A full-size launch returns in well under the kernel's 2 s bounded-wait
    limit with the error word clear: no wait of the kernel runs out."""
    import time
    case = kvgen.config_case("C1", device="cuda", kv_dtype=kv_dtype)
    kw = {} if kv_dtype == "bf16" else dict(k_scale=case.k_scale, v_scale=case.v_scale)
    run(cuda_lib, case, **kw)                 # warm-up (plan, tensor maps)
    t0 = time.perf_counter()
    for _ in range(5):
        run(cuda_lib, case, **kw)
    assert (time.perf_counter() - t0) / 5 < 0.2


@pytest.mark.parametrize("name", ["C1", "C2-MHA", "C2-MQA", "C4-GQA"])
def test_full_size_full_output(cuda_lib, name):
    """The named workloads at full size, in the launch configuration the
    benchmark uses: every (b, h) row of the output and of lse against the
    oracle."""
    case = kvgen.config_case(name, device="cuda")
    out, lse = run(cuda_lib, case)
    ref, lref = gqa_full_oracle(case)
    assert_attn_close(out, ref, name)
    assert_lse_close(lse, lref, name)


def test_mqa_vs_mha_workload(cuda_lib):
    """C2: the MQA result equals the MHA kernel run on the MQA K/V repeated
    32 times (shared q)."""
    case = kvgen.config_case("C2-MQA", device="cuda")
    out1, _ = run(cuda_lib, case)
    k_rep = case.k.expand(-1, 32, -1, -1).contiguous()
    v_rep = case.v.expand(-1, 32, -1, -1).contiguous()
    out2, _ = cuda_lib.gqa_decode(case.q, k_rep, v_rep, case.seqlens, scale=case.scale)
    torch.cuda.synchronize()
    assert_attn_close(out1, f64(out2), "C2 MQA vs MHA")


@pytest.mark.parametrize("kv_dtype,max_ctas", [("bf16", 2), ("bf16", 0), ("fp8", 2), ("fp8", 0)])
def test_lazy_rescale_heavy_tail(cuda_lib, kv_dtype, max_ctas):
    """Keys that line up with the first query head of their group at a few
    later positions, each stronger than the last: that head's running max
    jumps by 10-14 (base 2) at tiles past the first, in the token slots of
    every consumer warp, so each warp rescales O mid-sequence."""
    B, h, n_kv, d = 2, 8, 2, 128
    case = kvgen.gqa_case(B, h, n_kv, d, seqlens=[3000, 1100], seed=230, device="cuda")
    g = h // n_kv
    # positions in tiles 2, 9, 15, 30 of the first sequence (and the
    # in-range ones of the second), one in each warp's 16-token slice
    spikes = [(2 * 64 + 5, 1.0), (9 * 64 + 21, 2.0), (15 * 64 + 38, 3.0), (30 * 64 + 60, 4.0)]
    for b in range(B):
        for kv in range(n_kv):
            q0 = case.q[b, kv * g].float()
            for t, alpha in spikes:
                if t < int(case.seqlens[b]):
                    case.k[b, kv, t] = (alpha * q0).to(torch.bfloat16)
    kw = {}
    if kv_dtype == "fp8":
        # one scale per KV head from the values' own maxima (spikes included),
        # so the quantised spikes keep their size
        def quant(x):
            sc = (x.float().abs().amax(dim=(0, 2, 3)) / 448.0).clamp(min=1e-6)
            codes = (x.float() / sc.view(1, -1, 1, 1)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
            return codes.view(torch.uint8), sc.to(torch.float32)
        case.k, case.k_scale = quant(case.k)
        case.v, case.v_scale = quant(case.v)
        kw = dict(k_scale=case.k_scale, v_scale=case.v_scale)
        ref, lref = gqa_full_oracle(case)
    else:
        ref, lref = full_oracle(case)
    # the jumps are there: the first head's base-2 score at each spike
    # exceeds the running max before it by more than 8
    sc = f64(case.q[0, 0:1]) @ (oracle.dequant_e4m3(case.k.cpu().numpy(), case.k_scale.cpu().numpy())[0, 0]
                                if kv_dtype == "fp8" else f64(case.k[0, 0])).T
    s2 = (sc[0, :3000] * case.scale / np.log(2))
    jumps = [s2[t] - s2[:t].max() for t, _ in spikes[1:]]
    assert min(jumps) > 8.0, jumps
    out, lse = run(cuda_lib, case, max_ctas=max_ctas, **kw)
    assert_attn_close(out, ref, f"heavy tail {kv_dtype} max_ctas={max_ctas}")
    assert_lse_close(lse, lref)
