"""GPU parity of the FP8 (E4M3) K/V cache and the sliding-window ring cache
of kvdec_gqa_decode / kvdec_append_rope against the fp64 oracle, through the
C ABI ([ARG] "attention-variants-and-kv-cache" §六.3 and §五.3)."""
import numpy as np
import pytest
import torch

import kvgen
import oracle
from parity import assert_attn_close, assert_lse_close, f64, gqa_full_oracle

pytestmark = pytest.mark.gpu


def np_(t):
    return t.detach().to("cpu").numpy()


def run(kv, case, **kw):
    """One decode through the C ABI; a valid launch leaves the device error
    word clear."""
    flag = kv.new_error_flag()
    out, lse = kv.gqa_decode(case.q, case.k, case.v, case.seqlens, case.block_table,
                             scale=case.scale, k_scale=case.k_scale, v_scale=case.v_scale,
                             window=case.window, error_flag=flag, **kw)
    torch.cuda.synchronize()
    assert flag.item() == 0, f"device error word {flag.item():#x}"
    return out, lse


def full_oracle(case):
    bt = None if case.block_table is None else np_(case.block_table)
    sl = np_(case.seqlens)
    if case.k_scale is not None:
        return oracle.gqa_decode_fp8(f64(case.q), np_(case.k), np_(case.v), np_(case.k_scale),
                                     np_(case.v_scale), sl, case.scale, bt, case.window)
    return oracle.gqa_decode(f64(case.q), f64(case.k), f64(case.v), sl, case.scale, bt,
                             case.window)


FP8 = [
    # B, h, n_kv, seqlens, paged, max_ctas
    (3, 8, 2, [1, 65, 4000], False, 0),
    (6, 32, 8, [1, 63, 64, 65, 129, 1000], False, 0),
    (6, 32, 8, [1, 63, 64, 65, 129, 1000], False, 7),      # pieces merged across CTAs
    (4, 16, 16, [70, 300, 64, 5], False, 0),                # MHA
    (3, 32, 1, [33, 700, 1500], False, 3),                  # MQA, g = 32, few units: chunks of 16
    (2, 48, 1, [100, 260], False, 0),                       # g = 48: three head chunks of 16
    (160, 32, 1, [1 + (41 * i) % 300 for i in range(160)], False, 0),  # 160 units: two row tiles
    (3, 64, 8, [5000, 70, 1], True, 0),                     # 70B-shaped, paged
    (2, 16, 1, [129, 2000], True, 5),
    # group sizes below 8: the head rows fill part of the 8 MMA columns
    (4, 8, 4, [2, 128, 129, 3000], False, 0),               # g = 2
    (3, 12, 4, [1, 300, 2000], False, 5),                   # g = 3, pieces merged
    (2, 10, 2, [65, 900], True, 0),                         # g = 5, paged
    (2, 14, 2, [64, 1500], False, 3),                       # g = 7
]


@pytest.mark.parametrize("B,h,n_kv,sl,paged,max_ctas", FP8)
def test_fp8_full_parity(cuda_lib, B, h, n_kv, sl, paged, max_ctas):
    case = kvgen.gqa_case(B, h, n_kv, 128, seqlens=sl, paged=paged, seed=700 + B * h,
                          device="cuda", kv_dtype="fp8")
    out, lse = run(cuda_lib, case, max_ctas=max_ctas)
    ref, lref = full_oracle(case)
    assert_attn_close(out, ref, "out")
    assert_lse_close(lse, lref, "lse")


@pytest.mark.parametrize("max_ctas", [0, 7])
def test_fp8_large_capacity_takes_the_two_cta_form(cuda_lib, max_ctas):
    """A cache with room for more than 256 tiles per SM runs the transposed
    form's two-CTA build (six stages per CTA) instead of the three-CTA one.
    Here the block table is padded with unused columns, so the sequences stay
    short: the plan's grid, seen through the workspace size, shrinks, and the
    output still matches the oracle."""
    case = kvgen.gqa_case(4, 32, 8, 128, seqlens=[1, 65, 700, 3000], paged=True, seed=761,
                          device="cuda", kv_dtype="fp8")
    bt = case.block_table
    ws_short = cuda_lib.gqa_workspace_bytes(case.q, case.k, case.v, case.seqlens, bt)
    pad = torch.zeros((bt.shape[0], 2048 - bt.shape[1]), dtype=torch.int32, device="cuda")
    case.block_table = torch.cat([bt, pad], dim=1).contiguous()
    ws_long = cuda_lib.gqa_workspace_bytes(case.q, case.k, case.v, case.seqlens, case.block_table)
    assert ws_long < ws_short
    out, lse = run(cuda_lib, case, max_ctas=max_ctas)
    ref, lref = full_oracle(case)
    assert_attn_close(out, ref, "out")
    assert_lse_close(lse, lref, "lse")


def test_fp8_bf16_output_and_empty_sequence(cuda_lib):
    case = kvgen.gqa_case(3, 32, 8, 128, seqlens=[0, 300, 64], seed=705, device="cuda",
                          kv_dtype="fp8")
    out, lse = run(cuda_lib, case, out_dtype=torch.bfloat16)
    ref, lref = full_oracle(case)
    assert_attn_close(out, ref, "out")
    assert_lse_close(lse, lref, "lse")
    assert torch.all(out[0] == 0)


def test_fp8_scale_is_per_kv_head(cuda_lib):
    """Swapping two heads' scales moves those heads' outputs."""
    case = kvgen.gqa_case(2, 8, 2, 128, seqlens=[300, 90], seed=706, device="cuda",
                          kv_dtype="fp8")
    out, _ = run(cuda_lib, case)
    case.v_scale = case.v_scale.flip(0).contiguous()
    out2, _ = run(cuda_lib, case)
    assert not torch.allclose(out[:, :4], out2[:, :4], atol=1e-3)


@pytest.mark.parametrize("name", ["C1", "C4-GQA"])
def test_fp8_full_size_full_output(cuda_lib, name):
    """The Llama-3-8B-shaped and the long-context Llama-3-70B-shaped
    workloads with an E4M3 cache, in the launch configuration the benchmark
    times: every (b, h) row against the oracle's decode of the dequantised
    cache."""
    case = kvgen.config_case(name, device="cuda", kv_dtype="fp8")
    out, lse = run(cuda_lib, case)
    ref, lref = gqa_full_oracle(case)
    assert_attn_close(out, ref, name)
    assert_lse_close(lse, lref, name)


WIN = [
    # B, h, n_kv, seqlens, window, paged, fp8
    (4, 8, 2, [5, 100, 101, 1000], 100, False, False),
    (4, 32, 8, [64, 65, 3000, 1], 64, True, False),
    (3, 32, 8, [10, 500, 4096], 1000, False, True),
    (3, 16, 2, [7, 8, 9], 8, True, True),
    (2, 8, 1, [1, 77], 1, False, False),                     # only the newest token
    (3, 8, 2, [0, 20, 30], 200, False, False),               # all shorter than the window
]


@pytest.mark.parametrize("B,h,n_kv,sl,window,paged,fp8", WIN)
def test_window_parity(cuda_lib, B, h, n_kv, sl, window, paged, fp8):
    case = kvgen.gqa_case(B, h, n_kv, 128, seqlens=sl, paged=paged, seed=800 + window,
                          device="cuda", kv_dtype="fp8" if fp8 else "bf16", window=window)
    for mc in (0, 5):
        out, lse = run(cuda_lib, case, max_ctas=mc)
        ref, lref = full_oracle(case)
        assert_attn_close(out, ref, f"out max_ctas={mc}")
        assert_lse_close(lse, lref, f"lse max_ctas={mc}")


def code_order(c):
    c = c.astype(np.int64)
    return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)


@pytest.mark.parametrize("paged,window", [(False, 0), (True, 0), (False, 50), (True, 100)])
def test_fp8_append_parity(cuda_lib, paged, window):
    B, n_kv, d = 5, 2, 128
    sl = torch.tensor([0, 37, 64, 130, 1000], dtype=torch.int32)
    # a cache (random codes) whose table already covers the appended slot
    base = kvgen.gqa_case(B, 8, n_kv, d, seqlens=sl + 1, paged=paged, seed=900 + window,
                          kv_dtype="fp8", window=window)
    k_new, v_new = kvgen.append_inputs_gqa(B, n_kv, d, seed=901)
    bt = base.block_table
    K0, V0 = np_(base.k), np_(base.v)
    dev = "cuda"
    Kg, Vg = base.k.to(dev), base.v.to(dev)
    cuda_lib.append_rope_gqa(Kg, Vg, sl.to(dev), k_new.to(dev), v_new.to(dev),
                             None if bt is None else bt.to(dev),
                             k_scale=base.k_scale.to(dev), v_scale=base.v_scale.to(dev),
                             window=window)
    torch.cuda.synchronize()
    Kr, Vr = oracle.append_rope_gqa(
        K0, V0, np_(sl), np_(k_new.view(torch.int16)).view(np.uint16),
        np_(v_new.view(torch.int16)).view(np.uint16), None if bt is None else np_(bt),
        window=window, k_scale=np_(base.k_scale), v_scale=np_(base.v_scale))
    Kg, Vg = np_(Kg), np_(Vg)
    # V: the code is decided from the binary32 quotient on both sides (zero's
    # sign aside); K: the rotation's rounding may move a code by one step
    np.testing.assert_array_equal(code_order(Vg), code_order(Vr))
    assert np.abs(code_order(Kg) - code_order(Kr)).max() <= 1
    # nothing but the appended rows was written
    rows = np.any(Kr != K0, axis=-1) | np.any(Vr != V0, axis=-1)
    assert rows.sum() == B * n_kv
    np.testing.assert_array_equal(Kg[~rows], K0[~rows])
    np.testing.assert_array_equal(Vg[~rows], V0[~rows])


def test_ring_append_then_decode(cuda_lib):
    """Stream 150 tokens through a 100-slot ring, appending on the GPU one
    step at a time; then the decode over the ring equals the oracle's
    attention over the last 100 rotated keys appended by the oracle."""
    B, n_kv, d, h, w, N = 2, 2, 128, 8, 100, 150
    dev = "cuda"
    Kg = torch.zeros((B, n_kv, 128, d), dtype=torch.bfloat16, device=dev)
    Vg = torch.zeros_like(Kg)
    Kr = np.zeros((B, n_kv, 128, d), np.uint16)
    Vr = np.zeros((B, n_kv, 128, d), np.uint16)
    start = torch.tensor([0, 40], dtype=torch.int32)
    for step in range(N):
        sl = start + step
        k_new, v_new = kvgen.append_inputs_gqa(B, n_kv, d, seed=2000 + step)
        cuda_lib.append_rope_gqa(Kg, Vg, sl.to(dev), k_new.to(dev), v_new.to(dev), window=w)
        Kr, Vr = oracle.append_rope_gqa(Kr, Vr, np_(sl), np_(k_new.view(torch.int16)).view(np.uint16),
                                        np_(v_new.view(torch.int16)).view(np.uint16), window=w)
    torch.cuda.synchronize()
    total = (start + N).to(torch.int32)
    q = kvgen.gqa_case(B, h, n_kv, d, seqlens=[1, 1], seed=2999).q.to(dev)
    out, lse = cuda_lib.gqa_decode(q, Kg, Vg, total.to(dev), window=w)
    torch.cuda.synchronize()
    ref, lref = oracle.gqa_decode(f64(q), oracle.bf16_bits_to_f64(Kr), oracle.bf16_bits_to_f64(Vr),
                                  np_(total), 1 / np.sqrt(d), None, w)
    assert_attn_close(out, ref, "out")
    assert_lse_close(lse, lref, "lse")


def test_window_and_fp8_argument_errors(cuda_lib):
    case = kvgen.gqa_case(2, 8, 2, 128, seqlens=[10, 20], seed=5, device="cuda", kv_dtype="fp8")
    with pytest.raises(cuda_lib.KvdecError):
        cuda_lib.gqa_decode(case.q, case.k, case.v, case.seqlens, window=case.cap + 1,
                            k_scale=case.k_scale, v_scale=case.v_scale)
    p = cuda_lib.gqa_params(case.q, case.k, case.v, case.seqlens)   # no scales
    out = torch.empty(case.q.shape, device="cuda")
    p.out = out.data_ptr()
    ws = torch.zeros(cuda_lib.gqa_workspace_bytes(case.q, case.k, case.v, case.seqlens),
                     dtype=torch.uint8, device="cuda")
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    lib = cuda_lib.load()
    import ctypes
    assert lib.kvdec_gqa_decode(ctypes.byref(p), None) == 1
