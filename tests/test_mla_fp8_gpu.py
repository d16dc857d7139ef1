"""GPU parity of the E4M3 latent cache of kvdec_mla_decode_absorbed (the
widening pass, then the bf16 decode) and of the quantising MLA append
against the fp64 oracle, through the C ABI ([ARG]
"attention-variants-and-kv-cache" §六.3: FP8 halves the bytes of every
cached element; §四.5: the absorbed decode over [c_kv ; k_R] rows)."""
import ctypes
import time

import numpy as np
import pytest
import torch

import kvgen
import oracle
from parity import assert_attn_close, assert_lse_close, mla_full_oracle

pytestmark = pytest.mark.gpu


def np_(t):
    return t.detach().to("cpu").numpy()


def run(kv, case, **kw):
    """One decode through the C ABI; a valid launch leaves the device error
    word clear."""
    flag = kv.new_error_flag()
    out, lse = kv.mla_decode_absorbed(case.q_abs, case.q_rope, case.cache, case.block_table,
                                      case.seqlens, scale=case.scale, kv_scale=case.kv_scale,
                                      error_flag=flag, **kw)
    torch.cuda.synchronize()
    assert flag.item() == 0, f"device error word {flag.item():#x}"
    return out, lse


def fp8_case(sl, seed, **kw):
    return kvgen.mla_case(len(sl), 128, seqlens=sl, seed=seed, device="cuda", kv_dtype="fp8", **kw)


@pytest.mark.parametrize("sl", [[100, 700], [1, 64, 65], [64], [3000, 17, 129, 4096]])
def test_small_full_parity(cuda_lib, sl):
    case = fp8_case(sl, 300 + len(sl))
    out, lse = run(cuda_lib, case)
    ref, lref = mla_full_oracle(case)
    assert_attn_close(out, ref, "mla fp8")
    assert_lse_close(lse, lref, "mla fp8 lse")


def test_scales_are_used(cuda_lib):
    """Doubling the c_kv scale changes the result exactly as the oracle
    says, and so does a larger k_R scale (q_rope large enough that the rope
    term matters): the two scales are applied, to the right pieces.  The
    scales are powers of two, so the widened values are exact and the
    comparison isolates the scale routing from bf16 rounding."""
    def case_with(sc, sr):
        c = fp8_case([900, 333], 310)
        c.q_rope.mul_(4.0)
        c.kv_scale.copy_(torch.tensor([sc, sr], device="cuda"))
        return c
    base, _ = run(cuda_lib, case_with(2.0 ** -7, 2.0 ** -4))
    for sc, sr in [(2.0 ** -6, 2.0 ** -4), (2.0 ** -7, 2.0 ** -2)]:
        c2 = case_with(sc, sr)
        out, lse = run(cuda_lib, c2)
        ref, lref = mla_full_oracle(c2)
        assert_attn_close(out, ref, f"scales {sc}, {sr}")
        assert_lse_close(lse, lref)
        assert (out - base).abs().max().item() > 0.05


@pytest.mark.parametrize("max_ctas", [2, 6, 14, 0])
def test_split_invariance(cuda_lib, max_ctas):
    """Sequences cut across CTA pairs merge to the same result."""
    case = fp8_case([2500, 640, 5], 311)
    ref, lref = mla_full_oracle(case)
    out, lse = run(cuda_lib, case, max_ctas=max_ctas)
    assert_attn_close(out, ref, f"max_ctas={max_ctas}")
    assert_lse_close(lse, lref)


def test_empty_sequences_and_bf16(cuda_lib):
    case = fp8_case([0, 300, 0], 312)
    out, lse = run(cuda_lib, case, out_dtype=torch.bfloat16)
    assert out.dtype == torch.bfloat16
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    assert torch.isneginf(lse[0]).all() and torch.isneginf(lse[2]).all()
    ref, lref = mla_full_oracle(case)
    assert_attn_close(out, ref, "bf16 out")
    assert_lse_close(lse, lref)


def test_many_short_sequences(cuda_lib):
    """The largest batch the kernel takes, with the E4M3 layout's tile table
    filling its shared memory; some sequences are empty."""
    g = torch.Generator().manual_seed(6)
    sl = torch.randint(0, 200, (cuda_lib.load().kvdec_mla_max_batch(),), generator=g)
    sl[::41] = 0
    sl = sl.tolist()
    case = fp8_case(sl, 313)
    out, lse = run(cuda_lib, case)
    ref, lref = mla_full_oracle(case)
    assert_attn_close(out, ref, "many")
    assert_lse_close(lse, lref)


@pytest.mark.parametrize("max_ctas", [2, 0])
def test_lazy_rescale_heavy_tail(cuda_lib, max_ctas):
    """Heavy-tailed rope scores: the row maxima jump by more than 2^8 at
    random pages, so O is rescaled mid-sequence by both softmax groups."""
    case = fp8_case([3000, 1100], 314)
    g = torch.Generator(device="cuda").manual_seed(10)
    case.q_rope.zero_()
    case.q_rope[:, :, 0] = (1.5 * torch.randn((2, 128), generator=g, device="cuda")).to(torch.bfloat16)
    case.kv_scale[1] = 0.25
    spikes = torch.empty(case.cache.shape[:2], device="cuda").exponential_(1.0, generator=g)
    codes = (48.0 * spikes).clamp(max=448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    case.cache[:, :, 512] = codes
    out, lse = run(cuda_lib, case, max_ctas=max_ctas)
    ref, lref = mla_full_oracle(case)
    t = torch.arange(3000)
    k0 = oracle.e4m3_bits_to_f64(np_(case.cache.cpu()[case.block_table.cpu()[0, t // 64].long(), t % 64, 512]))
    k0 = k0 * 0.25
    sc = np_(case.q_rope[0, :, :1].double()) * k0[None, :] * case.scale / np.log(2)
    assert ((sc.max(1) - sc[:, :64].max(1)) > 8.0).any()
    assert_attn_close(out, ref, f"heavy tail, max_ctas={max_ctas}")
    assert_lse_close(lse, lref)


@pytest.mark.parametrize("name", ["C3", "C4-MLA"])
def test_full_size_full_output(cuda_lib, name):
    """The named workloads with an E4M3 cache, at full size in the launch
    configuration the benchmark uses: every (b, h) row of the output and of
    lse against the oracle."""
    case = kvgen.config_case(name, device="cuda", kv_dtype="fp8")
    out, lse = run(cuda_lib, case)
    ref, lref = mla_full_oracle(case)
    assert_attn_close(out, ref, name)
    assert_lse_close(lse, lref, name)


def test_launch_returns_promptly(cuda_lib):
    """A full-size call (widening + decode) ends well inside the decode's
    bounded-wait limit."""
    case = kvgen.config_case("C4-MLA", device="cuda", kv_dtype="fp8")
    run(cuda_lib, case)
    t0 = time.perf_counter()
    for _ in range(5):
        run(cuda_lib, case)
    assert (time.perf_counter() - t0) / 5 < 0.2


def code_order(c):
    c = c.astype(np.int64)
    return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)


def test_fp8_append_parity(cuda_lib):
    """Quantising MLA append against the oracle: c_kv codes bit-exact (both
    sides round the binary32 quotient), k_R codes within one code (the
    rotation's rounding), nothing else written."""
    sl = torch.tensor([0, 37, 64, 130, 1000], dtype=torch.int32)
    base = kvgen.mla_case(5, 128, seqlens=(sl + 1).tolist(), seed=320, spare_pages=3, kv_dtype="fp8")
    ckv, kr = kvgen.append_inputs_mla(5, seed=321)
    C0 = np_(base.cache)
    cg = base.cache.to("cuda")
    cuda_lib.append_rope_mla(cg, base.block_table.to("cuda"), sl.to("cuda"), ckv.to("cuda"), kr.to("cuda"),
                             kv_scale=base.kv_scale.to("cuda"))
    torch.cuda.synchronize()
    ref = oracle.append_rope_mla(C0, np_(base.block_table), np_(sl), np_(ckv.view(torch.int16)).view(np.uint16),
                                 np_(kr.view(torch.int16)).view(np.uint16), kv_scale=np_(base.kv_scale))
    got = np_(cg)
    np.testing.assert_array_equal(code_order(got[..., :512]), code_order(ref[..., :512]))
    assert np.abs(code_order(got[..., 512:]) - code_order(ref[..., 512:])).max() <= 1
    rows = np.any(ref != C0, axis=-1)
    assert rows.sum() == 5
    np.testing.assert_array_equal(got[~rows], C0[~rows])


def test_append_then_decode(cuda_lib):
    """Stream 70 tokens into an E4M3 cache on the GPU, one step at a time,
    then decode: the result equals the oracle's decode over the cache the
    oracle's own append built (k_R codes may differ by one step, within the
    tolerance)."""
    B, N = 2, 70
    start = [60, 1]
    case = kvgen.mla_case(B, 128, seqlens=[s + N for s in start], seed=330, kv_dtype="fp8")
    case.kv_scale = torch.tensor([0.01, 0.02], dtype=torch.float32)
    ref_cache = np_(case.cache)
    cg = case.cache.to("cuda")
    btg, ksg = case.block_table.to("cuda"), case.kv_scale.to("cuda")
    for step in range(N):
        sl = torch.tensor([s + step for s in start], dtype=torch.int32)
        ckv, kr = kvgen.append_inputs_mla(B, seed=3000 + step)
        cuda_lib.append_rope_mla(cg, btg, sl.to("cuda"), ckv.to("cuda"), kr.to("cuda"), kv_scale=ksg)
        ref_cache = oracle.append_rope_mla(ref_cache, np_(case.block_table), np_(sl),
                                           np_(ckv.view(torch.int16)).view(np.uint16),
                                           np_(kr.view(torch.int16)).view(np.uint16), kv_scale=np_(case.kv_scale))
    dev = kvgen.MlaCase(case.q_abs.to("cuda"), case.q_rope.to("cuda"), cg, case.seqlens.to("cuda"), btg,
                        case.scale, kv_scale=ksg)
    out, lse = run(cuda_lib, dev)
    ref, lref = oracle.mla_decode_absorbed_fp8(oracle.bf16_to_f64(case.q_abs), oracle.bf16_to_f64(case.q_rope),
                                               ref_cache, np_(case.kv_scale), np_(case.block_table),
                                               np_(case.seqlens), case.scale)
    assert_attn_close(out, ref, "append then decode")
    assert_lse_close(lse, lref)


def test_missing_scale_rejected(cuda_lib):
    """An E4M3 cache without its scales is rejected on the host."""
    case = fp8_case([100], 340)
    p = cuda_lib.mla_params(case.q_abs, case.q_rope, case.cache, case.block_table, case.seqlens,
                            out=torch.empty(case.q_abs.shape, device="cuda"))
    p.kv_scale = None
    lib = cuda_lib.load()
    ws = torch.empty(lib.kvdec_mla_workspace_bytes(ctypes.byref(p)), dtype=torch.uint8, device="cuda")
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    st = lib.kvdec_mla_decode_absorbed(ctypes.byref(p), None)
    assert st == 1 and "kv_scale" in lib.kvdec_last_error().decode()


def test_shared_pages(cuda_lib):
    """Two sequences over the same E4M3 pages with the same queries: the
    widening copies the pages once per reference and both rows agree."""
    case = fp8_case([700, 700], 341)
    case.block_table[1] = case.block_table[0]
    case.q_abs[1] = case.q_abs[0]
    case.q_rope[1] = case.q_rope[0]
    out, _ = run(cuda_lib, case)
    assert torch.equal(out[0], out[1])
    ref, _ = mla_full_oracle(case)
    assert_attn_close(out, ref, "shared pages")


def test_bad_page_reported(cuda_lib):
    """A block-table entry outside the cache sets the error bit; the page
    is read as zeros and the output stays finite."""
    case = fp8_case([200, 100], 342)
    case.block_table[0, 1] = case.cache.shape[0] + 3
    flag = cuda_lib.new_error_flag()
    out, _ = cuda_lib.mla_decode_absorbed(case.q_abs, case.q_rope, case.cache, case.block_table, case.seqlens,
                                          kv_scale=case.kv_scale, error_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() & cuda_lib.DEVERR_BAD_PAGE
    assert torch.isfinite(out).all()
