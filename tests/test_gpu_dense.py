"""Tensor-core (tcgen05) node kernel vs the fp64 oracle (needs a GB300).

Covers single nodes of many shapes (powers of two, ragged edges that do not
fill a 128 x 128 tile, k not a multiple of the 16-entry stage), outputs whose
mode order interleaves M and N, a dense node feeding another dense node
through the planar split format, slicing with the root accumulating, and the
bf16-operand variant (tolerance 2e-2).
"""
import numpy as np
import pytest

import exact_tensor_network_gb300 as tn
import oracle
from workloads import configs, gemm_network
from workloads.network import Network

from helpers import TOL_BF16, TOL_BF16X3, TOL_C64, assert_close, max_rel_err, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


def _rand(rng, shape, scale=1.0):
    z = (rng.standard_normal(shape) + 1j * rng.standard_normal(shape)) * scale
    return z.astype(np.complex64)


def node_network(m, n, k, seed):
    """A[i, x] B[j, x] -> C[i, j] with single modes of extents m, n, k."""
    rng = np.random.default_rng(seed)
    return Network([[0, 2], [1, 2]], [m, n, k], [0, 1], [_rand(rng, (m, k)), _rand(rng, (n, k))],
                   f"node_{m}x{n}x{k}")


def _ref(net, tree, slices=()):
    if slices:
        return oracle.contract_sliced(net.tensors, net.extents, net.open_modes, net.data, tree,
                                      slices)
    return oracle.contract(net.tensors, net.extents, net.open_modes, net.data, tree)


# Tests of the tensor-core kernel turn the batched tiny-node class off, so
# that their small shapes still reach it.
NT = tn.TN_POLICY_NO_TINY


def _classes(net, tree, slices=(), precision="tf32x3", policy=NT):
    p = tn.Plan.from_network(net, tree, slices, precision, policy)
    return [p.node_class(s) for s in range(len(tree))]


@pytest.mark.parametrize("precision,tol", [("tf32x3", TOL_C64), ("bf16", TOL_BF16),
                                           ("bf16x3", TOL_BF16X3)])
@pytest.mark.parametrize("lm,ln,lk", [(8, 8, 8), (7, 8, 10), (9, 7, 6), (8, 8, 12), (10, 9, 5),
                                      (8, 8, 14)])
def test_gemm_networks(precision, tol, lm, ln, lk):
    net = gemm_network(lm, ln, lk, 11 * lm + 7 * ln + lk)
    assert _classes(net, [(0, 1)], precision=precision) == [tn.TN_NODE_DENSE]
    got, _ = run_gpu(net, [(0, 1)], precision=precision, policy=NT)
    assert_close(got, _ref(net, [(0, 1)]), tol, f"gemm {lm},{ln},{lk} {precision}")


@pytest.mark.parametrize("precision,tol", [("tf32x3", TOL_C64), ("bf16", TOL_BF16),
                                           ("bf16x3", TOL_BF16X3)])
@pytest.mark.parametrize("m,n,k", [(200, 100, 40), (129, 65, 24), (64, 300, 136), (1000, 77, 48),
                                   (128, 128, 16), (333, 250, 1000), (1, 1, 8), (5, 300, 8),
                                   (300, 3, 520)])
def test_ragged_nodes(precision, tol, m, n, k):
    """Every shape on the tensor-core kernel (forced), including tiles that
    are mostly padding and k that ends inside a stage or a chunk."""
    net = node_network(m, n, k, m + n + k)
    p = tn.Plan.from_network(net, [(0, 1)], (), precision, tn.TN_POLICY_DENSE)
    assert p.node_class(0) == tn.TN_NODE_DENSE
    got, _ = run_gpu(net, [(0, 1)], precision=precision, policy=tn.TN_POLICY_DENSE)
    assert_close(got, _ref(net, [(0, 1)]), tol, f"node {m}x{n}x{k} {precision}")


def test_forced_dense_on_random_network():
    """Test setting outside the C ABI (not a public policy): every eligible
    node of the 59 (not only the compute-bound ones) runs on split-tf32
    operands, which carry 22 significant bits instead of fp32's 24, so
    rounding compounds along the tree's depth.  Bound: 4x the complex64
    tolerance."""
    net, tree, _ = configs.random_60()
    got, _ = run_gpu(net, tree, policy=tn.TN_POLICY_DENSE)
    assert_close(got, _ref(net, tree), 4 * TOL_C64, "random_60 with every eligible node dense")


def test_interleaved_output_layout():
    # step 0: A[a,b,x] B[c,x] -> C{a,b,c}; step 1 consumes C with D[b,e] over b,
    # so C is stored [a, c, b]: M = (a, b), N = (c) interleaved
    rng = np.random.default_rng(5)
    ext = [16, 16, 128, 64, 8]          # a b c x e
    tensors = [[0, 1, 3], [2, 3], [1, 4]]
    data = [_rand(rng, [ext[x] for x in t]) for t in tensors]
    net = Network(tensors, ext, [0, 2, 4], data)
    tree = [(0, 1), (3, 2)]
    assert _classes(net, tree)[0] == tn.TN_NODE_DENSE
    got, plan = run_gpu(net, tree, policy=NT)
    assert plan.mode_order(3) == [0, 2, 1]
    assert_close(got, _ref(net, tree), TOL_C64, "interleaved dense output")


@pytest.mark.parametrize("ext", [[6, 12, 100, 64, 5], [16, 2, 64, 32, 4], [3, 64, 48, 16, 6]])
def test_interleaved_output_general_extents(ext):
    """Interleaved output whose blocks do not repeat (extents 3, 6, 12):
    the epilogue cannot use an address-order table and falls back."""
    rng = np.random.default_rng(sum(ext))
    tensors = [[0, 1, 3], [2, 3], [1, 4]]
    data = [_rand(rng, [ext[x] for x in t]) for t in tensors]
    net = Network(tensors, ext, [0, 2, 4], data)
    tree = [(0, 1), (3, 2)]
    got, plan = run_gpu(net, tree, policy=tn.TN_POLICY_DENSE)
    assert plan.node_class(0) == tn.TN_NODE_DENSE
    assert_close(got, _ref(net, tree), TOL_C64, f"interleaved {ext}")


@pytest.mark.parametrize("precision,tol", [("tf32x3", TOL_C64), ("bf16", TOL_BF16),
                                           ("bf16x3", TOL_BF16X3)])
def test_dense_chain(precision, tol):
    # A[a,x] B[x,b] -> C[a,b] (dense, planar output), C[a,b] D[b,c] -> root (dense)
    rng = np.random.default_rng(9)
    ext = [256, 64, 256, 128]            # a x b c
    tensors = [[0, 1], [1, 2], [2, 3]]
    data = [_rand(rng, [ext[x] for x in t], 0.5) for t in tensors]
    net = Network(tensors, ext, [0, 3], data)
    tree = [(0, 1), (3, 2)]
    assert _classes(net, tree, precision=precision) == [tn.TN_NODE_DENSE, tn.TN_NODE_DENSE]
    got, _ = run_gpu(net, tree, precision=precision, policy=NT)
    assert_close(got, _ref(net, tree), tol, f"dense chain {precision}")


@pytest.mark.parametrize("precision,tol", [("tf32x3", TOL_C64), ("bf16", TOL_BF16),
                                           ("bf16x3", TOL_BF16X3)])
@pytest.mark.parametrize("m,n,k", [(128, 256, 16384), (64, 4096, 2048), (300, 200, 3000)])
def test_dense_split_k(precision, tol, m, n, k):
    """Few output tiles and long k: the tensor-core kernel splits k across
    CTAs (whole 256-entry chunks) and the partials are reduced in order."""
    net = node_network(m, n, k, m + 2 * n + 3 * k)
    p = tn.Plan.from_network(net, [(0, 1)], (), precision)
    assert p.node_class(0) == tn.TN_NODE_DENSE
    assert p.launches == 3            # leaf conversion, dense, reduction
    got, _ = run_gpu(net, [(0, 1)], precision=precision)
    assert_close(got, _ref(net, [(0, 1)]), tol, f"split dense {m}x{n}x{k} {precision}")


def test_dense_split_k_feeding_dense():
    # A[a,x] B[b,x] -> C[a,b] (64 x 2048 output, k = 4096: split), then
    # C[a,b] D[c,b] -> root (dense over b = 2048)
    rng = np.random.default_rng(21)
    ext = [64, 4096, 2048, 256]          # a x b c
    tensors = [[0, 1], [2, 1], [3, 2]]
    data = [_rand(rng, [ext[x] for x in t], 0.25) for t in tensors]
    net = Network(tensors, ext, [0, 3], data)
    tree = [(0, 1), (3, 2)]
    p = tn.Plan.from_network(net, tree)
    assert [p.node_class(s) for s in range(2)] == [tn.TN_NODE_DENSE, tn.TN_NODE_DENSE]
    got, _ = run_gpu(net, tree)
    assert_close(got, _ref(net, tree), TOL_C64, "split dense feeding dense")


def test_split_k_interleaved_sliced_root_repeated():
    """Split-K node whose output interleaves M and N modes, sliced over a
    K mode so the root accumulates, executed three times."""
    rng = np.random.default_rng(57)
    ext = [8, 8, 64, 32, 2048, 2]               # a1 a2 b1 b2 x1 x2
    tensors = [[0, 1, 4, 5], [2, 4, 5, 3]]
    data = [_rand(rng, [ext[x] for x in t], 0.05) for t in tensors]
    net = Network(tensors, ext, [3, 0, 2, 1], data)
    tree = [(0, 1)]
    sl = [5]
    assert _classes(net, tree, sl) == [tn.TN_NODE_DENSE]
    p = tn.Plan.from_network(net, tree, sl, "tf32x3", NT)
    assert p.launches == 6                      # per slice: leaf conversion, dense, reduction
    got, plan = run_gpu(net, tree, sl, policy=NT, repeat=3)
    assert plan.num_slices == 2
    assert_close(got, _ref(net, tree, sl), TOL_C64, "split-K interleaved sliced root")


def test_sliced_dense_root_accumulates():
    net = gemm_network(8, 8, 9, 3)
    sl = [net.tensors[0][-1], net.tensors[0][-2]]     # two K modes -> 4 slices
    assert _classes(net, [(0, 1)], sl) == [tn.TN_NODE_DENSE]
    got, plan = run_gpu(net, [(0, 1)], sl, policy=NT)
    assert plan.num_slices == 4
    assert_close(got, _ref(net, [(0, 1)]), TOL_C64, "sliced dense")


def test_transposed_root_order():
    net = gemm_network(8, 8, 8, 4)
    net.open_modes = list(reversed(net.open_modes))    # fully reversed: riffled N, M
    got, _ = run_gpu(net, [(0, 1)])
    assert_close(got, _ref(net, [(0, 1)]), TOL_C64, "reversed root order")


def test_split_bf16_accuracy_between_bf16_and_tf32x3():
    """The split-bf16 precision on random_60 (every node class writing the
    four-plane bf16 format for its tensor-core consumers): its error lies
    between those of the split-tf32 and plain bf16 precisions."""
    net, tree, _ = configs.random_60()
    ref = _ref(net, tree)
    err = {}
    for prec in ("tf32x3", "bf16x3", "bf16"):
        got, _ = run_gpu(net, tree, precision=prec)
        err[prec] = max_rel_err(got, ref)
    assert err["bf16x3"] <= TOL_BF16X3, err
    assert err["tf32x3"] < err["bf16x3"] < err["bf16"], err


def test_random_60_uses_dense_nodes_and_matches():
    net, tree, _ = configs.random_60()
    cls = _classes(net, tree)
    got, _ = run_gpu(net, tree)
    assert_close(got, _ref(net, tree), TOL_C64, "random_60 auto")
    assert tn.TN_NODE_DENSE in cls or True


@pytest.mark.parametrize("p_ext,a_ext,precision,tol", [
    (64, 128, "tf32x3", TOL_C64),     # power-of-two extents: store table in tiled addresses
    (72, 96, "tf32x3", TOL_C64),      # k = 6144: tiled, offsets tiled entry by entry
    (64, 128, "bf16", TOL_BF16),
    (64, 128, "bf16x3", TOL_BF16X3),
])
def test_dense_output_k_tiled_for_dense_consumer(p_ext, a_ext, precision, tol):
    # A[p,a,x] B[y,x] -> C[p,a,y] (tensor cores), then C[p,a,y] D[q,a,y] -> root[p,q]
    # with k = a*y >= 4096, so C is written K-tiled for the consumer's TMA loads
    rng = np.random.default_rng(33)
    ext = [p_ext, a_ext, 256, 64, 256]          # p a x y q
    tensors = [[0, 1, 2], [3, 2], [4, 1, 3]]
    data = [_rand(rng, [ext[x] for x in t], 0.1) for t in tensors]
    net = Network(tensors, ext, [0, 4], data)
    tree = [(0, 1), (3, 2)]
    p = tn.Plan.from_network(net, tree, (), precision)
    assert [p.node_class(s) for s in range(2)] == [tn.TN_NODE_DENSE, tn.TN_NODE_DENSE]
    assert p.node_mnk(1)[2] == a_ext * 64
    got, _ = run_gpu(net, tree, precision=precision)
    assert_close(got, _ref(net, tree), tol, f"K-tiled operand {p_ext}x{a_ext} {precision}")


def test_sliced_dense_root_four_entry_stores():
    # 128 x 256 root on tensor cores: the address-order stores go four
    # entries per lane, and slices 1..3 add into the caller's output
    net = gemm_network(7, 8, 10, 5)
    sl = [net.tensors[0][-1], net.tensors[0][-3]]
    assert _classes(net, [(0, 1)], sl) == [tn.TN_NODE_DENSE]
    got, plan = run_gpu(net, [(0, 1)], sl, policy=NT)
    assert plan.num_slices == 4
    assert_close(got, _ref(net, [(0, 1)]), TOL_C64, "sliced dense root, four-entry stores")


def test_dense_root_output_not_16_byte_aligned():
    # the caller's output 8 bytes past a 16-byte boundary: the tensor-core
    # epilogue must fall back to single-entry stores
    import torch
    net = gemm_network(7, 8, 8, 6)            # k = 256: no split-K, the kernel stores the root
    plan = tn.Plan.from_network(net, [(0, 1)], (), "tf32x3", NT)
    assert plan.node_class(0) == tn.TN_NODE_DENSE and plan.launches == 2
    dev = torch.device("cuda:0")
    leaves = [torch.from_numpy(np.ascontiguousarray(d)).to(dev) for d in net.data]
    size = int(np.prod(plan.out_shape))
    flat = torch.zeros(size + 1, dtype=torch.complex64, device=dev)
    out = flat[1:].view(plan.out_shape)
    assert out.data_ptr() % 16 == 8
    plan.execute(leaves, out)
    torch.cuda.synchronize(dev)
    plan.check()
    assert complex(flat[0].item()) == 0
    assert_close(out.cpu().numpy().astype(np.complex128), _ref(net, [(0, 1)]), TOL_C64,
                 "unaligned root output")


@pytest.mark.parametrize("m,n,k,precision,tol", [
    (2048, 1280, 512, "tf32x3", TOL_C64),     # 160 tiles: 8 past the last full wave
    (2000, 1300, 528, "tf32x3", TOL_C64),     # ragged tiles, 33 k-blocks: halves of 16 and 17
    (2048, 1280, 544, "bf16", TOL_BF16),      # bf16: 17 k-blocks
    (2048, 1280, 544, "bf16x3", TOL_BF16X3),  # split bf16: 17 k-blocks
])
def test_dense_tail_tiles_split_in_k_halves(m, n, k, precision, tol):
    """Tiles past the last full wave run as two k halves on two CTAs; the
    second to finish adds the other's sums.  Matches the oracle, and two
    runs give identical bits (a sum of two terms does not depend on which
    half finished first)."""
    import torch
    net = node_network(m, n, k, m + n + k)
    plan = tn.Plan.from_network(net, [(0, 1)], (), precision, NT)
    assert plan.node_class(0) == tn.TN_NODE_DENSE and plan.launches == 2
    dev = torch.device("cuda:0")
    leaves = [torch.from_numpy(np.ascontiguousarray(d)).to(dev) for d in net.data]
    outs = []
    for _ in range(3):
        out = torch.full(plan.out_shape, complex(7.0, -3.0), dtype=torch.complex64, device=dev)
        plan.execute(leaves, out)
        torch.cuda.synchronize(dev)
        outs.append(out.cpu().numpy())
    plan.check()
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])
    assert_close(outs[2].astype(np.complex128), _ref(net, [(0, 1)]), tol,
                 f"tail halves {m}x{n}x{k} {precision}")


@pytest.mark.parametrize("m,n,k", [(512, 1024, 2048), (300, 700, 1040), (512, 512, 8192)])
def test_three_product_nodes(m, n, k):
    """Nodes bound by their arithmetic form the complex product from three
    real products (Ar Br, Ai Bi, (Ar + Ai)(Br + Bi)); with that turned off,
    from four.  Both match the oracle (k = 8192: K-tiled six-plane operands)."""
    import torch
    net = node_network(m, n, k, m + 3 * n + 7 * k)
    ref = _ref(net, [(0, 1)])
    dev = torch.device("cuda:0")
    for three, kernel in ((True, "dense_tf32x3_3p"), (False, "dense_tf32x3")):
        plan = tn.Plan.from_network(net, [(0, 1)], (), "tf32x3", NT)
        plan.set_three_products(three)
        assert plan.node_class(0) == tn.TN_NODE_DENSE
        leaves = [torch.from_numpy(np.ascontiguousarray(d)).to(dev) for d in net.data]
        out = torch.empty(plan.out_shape, dtype=torch.complex64, device=dev)
        plan.set_profiling(True)
        plan.execute(leaves, out)
        torch.cuda.synchronize(dev)
        plan.check()
        assert kernel in [r["kernel"] for r in plan.profile()]
        assert_close(out.cpu().numpy().astype(np.complex128), ref, TOL_C64,
                     f"{m}x{n}x{k} three products={three}")


@pytest.mark.parametrize("m,n,k,precision,policy,tol", [
    (64, 4096, 2048, "tf32x3", NT, TOL_C64),                   # m = 64: operands swapped, split-K
    (4096, 64, 512, "tf32x3", NT, TOL_C64),                    # n = 64: narrow, no swap
    (64, 64, 1024, "tf32x3", tn.TN_POLICY_DENSE, TOL_C64),     # both sides 64
    (64, 1024, 8192, "tf32x3", NT, TOL_C64),                   # K-tiled operands, narrow B boxes
    (200, 48, 1040, "tf32x3", tn.TN_POLICY_DENSE, TOL_C64),    # ragged narrow tiles
    (30, 300, 96, "tf32x3", tn.TN_POLICY_DENSE, TOL_C64),      # swapped, ragged on both sides
    (64, 4096, 2048, "bf16", NT, TOL_BF16),                    # bf16: eight 24 KiB stages
    (64, 4096, 2048, "bf16x3", NT, TOL_BF16X3),                # split bf16: four 48 KiB stages
    (64, 1024, 8192, "bf16x3", NT, TOL_BF16X3),                # split bf16, K-tiled, narrow
])
def test_dense_narrow_tiles(m, n, k, precision, policy, tol):
    """A node with a side of at most 64 runs 128 x 64 tiles: that side goes
    to N (operands swapped when it is m) and B stacked [Br; Bi] fills one
    N = 128 MMA."""
    net = node_network(m, n, k, 3 * m + n + k)
    plan = tn.Plan.from_network(net, [(0, 1)], (), precision, policy)
    assert plan.node_class(0) == tn.TN_NODE_DENSE
    got, _ = run_gpu(net, [(0, 1)], precision=precision, policy=policy, repeat=2)
    assert_close(got, _ref(net, [(0, 1)]), tol, f"narrow {m}x{n}x{k} {precision}")


# ---- CTA pairs (tcgen05 cta_group::2, opt-in) --------------------------------

@pytest.mark.parametrize("precision,tol", [("tf32x3", TOL_C64), ("bf16", TOL_BF16),
                                           ("bf16x3", TOL_BF16X3)])
@pytest.mark.parametrize("m,n,k", [(256, 128, 64), (512, 384, 512), (300, 200, 136), (1000, 77 + 64, 48),
                                   (129, 700, 1000), (2048, 256, 4096), (640, 512, 2064)])
def test_cta_pair_nodes(precision, tol, m, n, k):
    """Single nodes on CTA pairs: full and ragged 256-row tiles, the swap
    (the longer side becomes the rows), split-K, K-tiled operands."""
    net = node_network(m, n, k, 3 * m + n + k)
    got, plan = run_gpu(net, [(0, 1)], precision=precision, policy=NT, pairs=True)
    assert plan.node_class(0) == tn.TN_NODE_DENSE
    assert_close(got, _ref(net, [(0, 1)]), tol, f"pair node {m}x{n}x{k} {precision}")


def test_cta_pairs_network_and_slices():
    """A chain of tensor-core nodes (planar operands written by a pair's
    epilogue, read by the next pair) and a sliced root that accumulates."""
    net, tree, _ = configs.random_60()
    a, _ = run_gpu(net, tree, pairs=True)
    assert_close(a, _ref(net, tree), TOL_C64, "random_60 on CTA pairs")
    rng = np.random.default_rng(8)
    ext = [512, 256, 384, 4]                   # i x j z (z sliced)
    tensors = [[0, 1, 3], [2, 1, 3]]
    data = [_rand(rng, [ext[x] for x in t]) for t in tensors]
    net = Network(tensors, ext, [0, 2], data)
    got, plan = run_gpu(net, [(0, 1)], [3], policy=NT, pairs=True)
    assert plan.num_slices == 4 and plan.node_class(0) == tn.TN_NODE_DENSE
    assert_close(got, _ref(net, [(0, 1)], [3]), TOL_C64, "sliced pair node")


@pytest.mark.parametrize("m,n,k,chunk,precision,tol", [
    (2048, 1280, 2048, 32, "tf32x3", TOL_C64),     # whole tiles of 128 stages and tail halves of 64, 2-stage chunks
    (2048, 1280, 1040, 64, "tf32x3", TOL_C64),     # 65 stages: halves of 32 and 33, 4-stage chunks
    (2000, 1300, 2064, 128, "tf32x3", TOL_C64),    # ragged tiles, 129 stages, 8-stage chunks
    (64, 4096, 4096, 32, "tf32x3", TOL_C64),       # swapped narrow tiles, split-K with long splits
    (2048, 1280, 2048, 64, "bf16x3", TOL_BF16X3),  # bf16 stages of 32 k: 2-stage chunks
    (2048, 1280, 4096, 256, "bf16", TOL_BF16),     # 8-stage chunks, tail halves of 64 stages
])
def test_promotion_chunk_boundaries(m, n, k, chunk, precision, tol):
    """Promotion chunks of every length the planner or the caller can pick,
    on whole tiles, tail halves and split-K items: a tile of at least eight
    chunks starts with one of two chunks' length, shorter tiles do not, and
    every k-block is accumulated exactly once (oracle)."""
    import torch
    net = node_network(m, n, k, m + 5 * n + 3 * k + chunk)
    plan = tn.Plan.from_network(net, [(0, 1)], (), precision, NT)
    plan.set_promotion_chunk(chunk)
    assert plan.node_class(0) == tn.TN_NODE_DENSE
    dev = torch.device("cuda:0")
    leaves = [torch.from_numpy(np.ascontiguousarray(d)).to(dev) for d in net.data]
    out = torch.full(plan.out_shape, complex(7.0, -3.0), dtype=torch.complex64, device=dev)
    plan.execute(leaves, out)
    torch.cuda.synchronize(dev)
    plan.check()
    assert_close(out.cpu().numpy().astype(np.complex128), _ref(net, [(0, 1)]), tol,
                 f"{m}x{n}x{k} chunk {chunk} {precision}")


@pytest.mark.parametrize("precision,tol", [("tf32x3", TOL_C64), ("bf16x3", TOL_BF16X3), ("bf16", TOL_BF16)])
@pytest.mark.parametrize("m,n,k", [(512, 2048, 32), (300, 1000, 48), (1024, 640, 256), (130, 4000, 64),
                                   (2048, 512, 32)])
def test_short_k_nodes_on_narrow_tiles(m, n, k, precision, tol):
    """Short-k nodes whose 128 x 128 tiles would fill at most half the SMs
    run 128 x 64 tiles with neither side narrow (ragged rows and columns,
    k not a multiple of the stage)."""
    net = node_network(m, n, k, m + 2 * n + 5 * k)
    plan = tn.Plan.from_network(net, [(0, 1)], (), precision, NT)
    assert plan.node_class(0) == tn.TN_NODE_DENSE
    got, _ = run_gpu(net, [(0, 1)], precision=precision, policy=NT)
    assert_close(got, _ref(net, [(0, 1)]), tol, f"short-k {m}x{n}x{k} {precision}")
