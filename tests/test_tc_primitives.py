"""Each tcgen05 operand form the attention kernels use, checked alone on one
128x128x128 bf16 product (fp32 accumulation) against an fp64 matmul of the
same bf16 values."""
import pytest
import torch

from long_context_causal_gb300 import dfa

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("form", [0, 1, 2, 3])
def test_mma_form(form):
    g = torch.Generator(device="cuda").manual_seed(100 + form)
    A = torch.randn((128, 128), generator=g, device="cuda").to(torch.bfloat16)
    B = torch.randn((128, 128), generator=g, device="cuda").to(torch.bfloat16)
    C = dfa.dfa_debug_mma(form, A, B)
    dfa.dfa_check_errors()
    a, b = A.double(), B.double()
    ref = {0: a @ b.T, 1: a @ b, 2: a.T @ b, 3: a @ b.T}[form]
    err = (C.double() - ref).abs().max().item()
    assert err < 1e-3, f"form {form}: max abs err {err}"
