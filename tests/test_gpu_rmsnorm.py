"""GPU numerics of eagle3_rmsnorm (w * x * rsqrt(mean(x^2) + eps)) against fp64, the embedding
gather and the aux-tap copy (bit-exact)."""
import numpy as np
import pytest
import torch

from tests._util import close, require_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,dim", [(1, 64), (7, 4096), (300, 4096), (5, 100), (64, 12288)])
def test_rmsnorm(rows, dim):
    from eagle_tree_speculative_spec_gb300 import eagle3_rmsnorm
    dev = require_gpu()
    g = torch.Generator().manual_seed(rows + dim)
    x = (3 * torch.randn(rows, dim, generator=g)).to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn(dim, generator=g)).to(torch.bfloat16)
    out = torch.empty(rows, dim, dtype=torch.bfloat16, device=dev)
    tap = torch.empty(rows, dim, dtype=torch.bfloat16, device=dev)
    eagle3_rmsnorm(x.to(dev), w.to(dev), out, eps=1e-5, tap_out=tap)
    torch.cuda.synchronize()
    xd = x.double().numpy()
    ref = w.double().numpy() * xd / np.sqrt((xd * xd).mean(-1, keepdims=True) + 1e-5)
    ok, err = close(out.float().cpu().numpy(), ref, 2e-2, 1e-2)
    assert ok, err
    assert torch.equal(tap.cpu(), x)


def test_rmsnorm_gather_and_strided_tap():
    from eagle_tree_speculative_spec_gb300 import eagle3_rmsnorm
    dev = require_gpu()
    V, d, rows = 1000, 256, 37
    g = torch.Generator().manual_seed(3)
    table = torch.randn(V, d, generator=g).to(torch.bfloat16)
    w = torch.ones(d, dtype=torch.bfloat16)
    ids = torch.randint(0, V, (rows,), generator=g, dtype=torch.int32)
    out = torch.empty(rows, d, dtype=torch.bfloat16, device=dev)
    aux = torch.zeros(rows, 3 * d, dtype=torch.bfloat16, device=dev)
    eagle3_rmsnorm(table.to(dev), w.to(dev), out, gather=ids.to(dev), tap_out=aux[:, d:2 * d])
    torch.cuda.synchronize()
    rows_x = table[ids.long()]
    assert torch.equal(aux[:, d:2 * d].cpu(), rows_x)
    assert float(aux[:, :d].abs().sum()) == 0.0 and float(aux[:, 2 * d:].abs().sum()) == 0.0
    xd = rows_x.double().numpy()
    ref = xd / np.sqrt((xd * xd).mean(-1, keepdims=True) + 1e-5)
    ok, err = close(out.float().cpu().numpy(), ref, 2e-2, 1e-2)
    assert ok, err
