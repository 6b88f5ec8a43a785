"""Shared helpers for the GPU parity tests: run a network through the C ABI
and compare with the oracle element by element."""
import numpy as np

TOL_C64 = 1e-5     # max |gpu - ref| <= TOL * max |ref| for complex64 paths
TOL_BF16 = 2e-2    # bf16 tensor-core operands
# split bf16 (hi + lo keep 16 significant bits; lo*lo dropped): at most
# 3 * 2^-16 = 4.6e-5 of |a||b| per product, random-signed over k, and
# compounded through a chain of nodes
TOL_BF16X3 = 2e-4


def run_gpu(net, tree, slices=(), precision="tf32x3", policy=0, out_dtype=None, repeat=1):
    import torch
    import exact_tensor_network_gb300 as tn
    dev = torch.device("cuda:0")
    plan = tn.Plan.from_network(net, tree, slices, precision, policy)
    leaves = [torch.from_numpy(np.ascontiguousarray(d)).to(dev) for d in net.data]
    out = torch.full(plan.out_shape, complex(7.0, -3.0), dtype=torch.complex64, device=dev)
    for _ in range(repeat):
        plan.execute(leaves, out)
    torch.cuda.synchronize(dev)
    plan.check()
    return out.cpu().numpy().astype(np.complex128), plan


def node_network(m, n, k, seed, name=None):
    """Single step A[i, x] B[j, x] -> C[i, j] with one mode per side
    (extents m, n, k; a side of extent 1 still gets its mode)."""
    from workloads.network import Network
    rng = np.random.default_rng(seed)

    def rnd(shape):
        return ((rng.standard_normal(shape) + 1j * rng.standard_normal(shape))
                .astype(np.complex64))
    return Network([[0, 2], [1, 2]], [m, n, k], [0, 1], [rnd((m, k)), rnd((n, k))],
                   name or f"node_{m}x{n}x{k}")


def max_rel_err(got, ref):
    scale = float(np.abs(ref).max()) if np.size(ref) else 0.0
    err = float(np.abs(np.asarray(got) - np.asarray(ref)).max()) if np.size(ref) else 0.0
    return err / scale if scale > 0 else err


def assert_close(got, ref, tol=TOL_C64, what=""):
    assert np.shape(got) == np.shape(ref), (np.shape(got), np.shape(ref))
    r = max_rel_err(got, ref)
    assert r <= tol, f"{what}: max|err|/max|ref| = {r:.3e} > {tol:.1e}"
