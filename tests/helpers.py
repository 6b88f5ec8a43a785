"""Shared helpers for the GPU parity tests: run a network through the C ABI
and compare with the oracle element by element."""
import numpy as np

TOL_C64 = 1e-5     # max |gpu - ref| <= TOL * max |ref| for complex64 paths
TOL_BF16 = 2e-2    # bf16 tensor-core operands
# split bf16 (hi + lo keep 16 significant bits; lo*lo dropped): at most
# 3 * 2^-16 = 4.6e-5 of |a||b| per product, random-signed over k, and
# compounded through a chain of nodes
TOL_BF16X3 = 2e-4


def run_gpu(net, tree, slices=(), precision="tf32x3", policy=0, out_dtype=None, repeat=1,
            fuse=True, pairs=False):
    import torch
    import exact_tensor_network_gb300 as tn
    dev = torch.device("cuda:0")
    plan = tn.Plan.from_network(net, tree, slices, precision, policy)
    if not fuse:
        plan.set_fusion(False)
    if pairs:
        plan.set_cta_pairs(True)
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


def node_layout(plan, step, extents):
    """(a, b, out, m, n, k, offM, offN) of a step from the plan's mode
    orders: A = [M | K] and B = [N | K] row-major, and the offset of output
    entry (i, j) in the output's own order is offM(i) + offN(j)."""
    n_leaves = plan.n_tensors
    a, b = plan.pairs[step]
    out = n_leaves + step
    oa, ob, oc = plan.mode_order(a), plan.mode_order(b), plan.mode_order(out)
    M = [x for x in oa if x not in ob]
    N = [x for x in ob if x not in oa]
    K = oa[len(M):]
    assert K == ob[len(N):], "operands must share the K order"
    assert sorted(oc) == sorted(M + N)
    ext = {x: int(extents[x]) for x in oa + ob}

    def prod(xs):
        r = 1
        for x in xs:
            r *= ext[x]
        return r
    stride_c = {}
    acc = 1
    for x in reversed(oc):
        stride_c[x] = acc
        acc *= ext[x]

    def side_offsets(side, idx):
        idx = np.asarray(idx, dtype=np.int64)
        off = np.zeros_like(idx)
        for x in reversed(side):
            off += (idx % ext[x]) * stride_c[x]
            idx = idx // ext[x]
        return off
    return (a, b, out, prod(M), prod(N), prod(K),
            lambda i: side_offsets(M, i), lambda j: side_offsets(N, j))


def check_node_sampled(plan, extents, leaves, out, step, seed, rows=64, cols=16, tol=TOL_C64):
    """Run the first slice up to `step` (tn_execute_prefix), read `rows`
    sampled rows of A, `cols` rows of B and the rows x cols outputs they
    give (tn_plan_tensor_gather), and compare those outputs with fp64 dot
    products of the gathered operand rows.  Returns the relative error."""
    import torch
    dev = out.device
    a, b, c, m, n, k, offm, offn = node_layout(plan, step, extents)
    rng = np.random.default_rng(seed)
    I = np.unique(rng.integers(0, m, size=min(rows, m)))
    J = np.unique(rng.integers(0, n, size=min(cols, n)))
    plan.execute_prefix(leaves, out, step)
    kk = np.arange(k, dtype=np.int64)

    def gather(t, idx):
        g = plan.gather(t, torch.from_numpy(np.ascontiguousarray(idx.ravel())).to(dev))
        return g.cpu().numpy().astype(np.complex128).reshape(idx.shape)
    A = gather(a, I[:, None] * k + kk[None, :])
    B = gather(b, J[:, None] * k + kk[None, :])
    C = gather(c, offm(I)[:, None] + offn(J)[None, :])
    torch.cuda.synchronize(dev)
    plan.check()
    ref = A @ B.T
    return max_rel_err(C, ref), (m, n, k)
