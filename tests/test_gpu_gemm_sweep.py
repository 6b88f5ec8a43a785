"""Single-node sweep at full size (needs a GB300 with ~230 GB free).

Two leaves with dimension-2 modes, A = [M||K], B = [N||K], result [M||N],
m, n, k each in {2^8, 2^12, 2^16} (27 shapes), complex64 N(0,1) entries,
in both tensor-core precisions.  The largest shape holds 32 GiB per
operand.  Checks, since the fp64 oracle cannot do 2^48 multiply-adds:
  * 1024 sampled outputs against fp64 dot products of the same leaves;
  * a Freivalds projection over every output: C x against A (B^T x) in
    fp64 for a random complex x.
Tolerances: 1e-5 x max|ref| (tf32x3), 2e-2 (bf16 operands).
"""
import itertools

import numpy as np
import pytest

import exact_tensor_network_gb300 as tn
from workloads import gemm_network

from helpers import TOL_BF16, TOL_C64, max_rel_err

pytestmark = pytest.mark.gpu

SHAPES = list(itertools.product((8, 12, 16), repeat=3))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("precision", ["tf32x3", "bf16"])
@pytest.mark.parametrize("lm,ln,lk", SHAPES)
def test_gemm_full_size(precision, lm, ln, lk):
    import torch
    tol = TOL_C64 if precision == "tf32x3" else TOL_BF16
    m, n, k = 1 << lm, 1 << ln, 1 << lk
    net = gemm_network(lm, ln, lk, 0, with_data=False)
    plan = tn.Plan.from_network(net, [(0, 1)], (), precision)
    assert plan.node_class(0) == tn.TN_NODE_DENSE
    dev = torch.device("cuda:0")
    torch.cuda.empty_cache()
    gen = torch.Generator(device=dev)
    gen.manual_seed(lm * 100 + ln * 10 + lk)
    A = torch.randn((m, k), dtype=torch.complex64, device=dev, generator=gen)
    B = torch.randn((n, k), dtype=torch.complex64, device=dev, generator=gen)
    C = torch.empty((m, n), dtype=torch.complex64, device=dev)
    plan.execute([A, B], C)
    torch.cuda.synchronize()
    plan.check()
    plan = None                      # release the workspace
    torch.cuda.empty_cache()
    rng = np.random.default_rng(lm + ln + lk)
    rows = torch.from_numpy(rng.integers(0, m, size=1024)).to(dev)
    cols = torch.from_numpy(rng.integers(0, n, size=1024)).to(dev)
    ref = (A[rows].to(torch.complex128) * B[cols].to(torch.complex128)).sum(dim=1)
    got = C[rows, cols].to(torch.complex128)
    r = max_rel_err(got.cpu().numpy(), ref.cpu().numpy())
    assert r <= tol, f"sampled: {r:.3e}"
    # Freivalds: C x = A (B^T x), every output entry enters the projection
    x = torch.randn(n, dtype=torch.complex128, device=dev, generator=gen)
    btx = torch.zeros(k, dtype=torch.complex128, device=dev)
    for j0 in range(0, n, 4096):
        btx += B[j0:j0 + 4096].to(torch.complex128).T @ x[j0:j0 + 4096]
    lhs = torch.empty(m, dtype=torch.complex128, device=dev)
    rhs = torch.empty(m, dtype=torch.complex128, device=dev)
    for i0 in range(0, m, 4096):
        lhs[i0:i0 + 4096] = C[i0:i0 + 4096].to(torch.complex128) @ x
        rhs[i0:i0 + 4096] = A[i0:i0 + 4096].to(torch.complex128) @ btx
    r2 = max_rel_err(lhs.cpu().numpy(), rhs.cpu().numpy())
    assert r2 <= tol, f"Freivalds: {r2:.3e}"
    del A, B, C
    torch.cuda.empty_cache()
