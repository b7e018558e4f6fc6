"""The LM-head GEMM with its row-statistics epilogue (include/headloss_lmhead.h)
on the GPU: logits against torch's matmul rounded once to bf16, and the
per-tile statistics against the same quantities computed from the kernel's
own bf16 logits.  Shapes: one tile with one K block, and 2 x 2 tiles with
two K blocks."""
import pytest
import torch

from gradient_row_online_gb300 import headloss as hlb

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,D,V", [(128, 64, 256), (256, 128, 512)])
def test_lmhead_logits_and_tile_statistics(N, D, V):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    hid = (torch.randn(N, D, generator=g, device="cuda") * 0.5).to(torch.bfloat16)
    wt = (torch.randn(V, D, generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    out = torch.zeros(N, V, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(N, V // 256, 2, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hlb.headloss_lmhead_logits(hid, wt, N, D, V, out, st, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = (hid.double() @ wt.double().T).to(torch.bfloat16).double()
    # fp32 accumulation in another order: at most one bf16 step from the
    # correctly rounded value
    d = (out.double() - ref).abs()
    assert bool((d <= ref.abs() * 2.0 ** -7 + 1e-6).all()), float(d.max())
    x = out.double().view(N, V // 256, 256)
    m = x.max(-1).values
    s = torch.exp(x - m[..., None]).sum(-1)
    assert torch.equal(st[..., 0].double(), m)
    assert float(((st[..., 1].double() - s) / s).abs().max()) < 1e-5
