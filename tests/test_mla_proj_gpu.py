"""GPU parity of the two MLA absorption projections (kvdec_mla_absorb_q,
kvdec_mla_project_out) and of a whole MLA attention layer built from them
and the absorbed decode, against the fp64 oracle, through the C ABI."""
import pytest
import torch

import kvgen
import oracle
from parity import assert_attn_close, f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H", [(1, 128), (7, 128), (64, 128), (130, 4), (3, 1)])
def test_absorb_q(cuda_lib, B, H):
    q_nope, W_UK, _ = kvgen.mla_proj_case(B, H, seed=300 + B, device="cuda")
    out = cuda_lib.mla_absorb_q(q_nope, W_UK, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = oracle.mla_absorb_q(f64(q_nope), f64(W_UK))
    assert_attn_close(out, ref, f"absorb B={B} H={H}", atol=2e-3, row_rtol=1e-3)
    outb = cuda_lib.mla_absorb_q(q_nope, W_UK)
    torch.cuda.synchronize()
    assert outb.dtype == torch.bfloat16
    assert_attn_close(outb, ref, f"absorb bf16 B={B} H={H}")


@pytest.mark.parametrize("B,H", [(1, 128), (9, 128), (64, 128), (65, 2)])
def test_project_out(cuda_lib, B, H):
    _, _, W_UV = kvgen.mla_proj_case(B, H, seed=310 + B, device="cuda")
    lat = kvgen.mla_proj_case(B, H, seed=320 + B, device="cuda")[0].repeat(1, 1, 4).contiguous()
    out = cuda_lib.mla_project_out(lat, W_UV)
    torch.cuda.synchronize()
    ref = oracle.mla_project_out(f64(lat), f64(W_UV))
    assert_attn_close(out, ref, f"project B={B} H={H}", atol=2e-3, row_rtol=1e-3)


def test_attention_layer_end_to_end(cuda_lib):
    """absorb -> absorbed decode (bf16 latent) -> project equals the literal
    non-absorbed MLA attention of the oracle ([ARG] §四.5, [MLA] §4)."""
    case = kvgen.mla_case(3, 128, seqlens=[700, 64, 1500], seed=330, device="cuda")
    q_nope, W_UK, W_UV = kvgen.mla_proj_case(3, 128, seed=331, device="cuda")
    q_abs = cuda_lib.mla_absorb_q(q_nope, W_UK)
    lat, _ = cuda_lib.mla_decode_absorbed(q_abs, case.q_rope, case.cache, case.block_table, case.seqlens,
                                          scale=case.scale, out_dtype=torch.bfloat16)
    out = cuda_lib.mla_project_out(lat, W_UV)
    torch.cuda.synchronize()
    ref, _ = oracle.mla_decode_nonabsorbed(f64(q_nope), f64(case.q_rope), f64(case.cache),
                                           case.block_table.cpu().numpy(), case.seqlens.cpu().numpy(),
                                           f64(W_UK), f64(W_UV), case.scale)
    assert_attn_close(out, ref, "MLA layer")
