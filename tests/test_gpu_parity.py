"""GPU path vs the fp64 oracle, element by element (needs a GB300).

Every case goes through the C ABI (tn_plan / tn_plan_set_workspace /
tn_execute) on seeded synthetic inputs and is compared with the oracle on the
same inputs: max |gpu - ref| <= 1e-5 * max |ref| for complex64 arithmetic.
"""
import numpy as np
import pytest

import oracle
from oracle.statevector import amplitudes
from workloads import (choose_slices, configs, gemm_network, greedy_tree, grid_circuit_network,
                       largest_intermediate, random_network, random_tiny_network)
from workloads.network import Network

from helpers import TOL_C64, assert_close, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


def _ref(net, tree, slices=()):
    if slices:
        return oracle.contract_sliced(net.tensors, net.extents, net.open_modes, net.data, tree, slices)
    return oracle.contract(net.tensors, net.extents, net.open_modes, net.data, tree)


def test_circuit_3x3_d4_amplitude():
    net, tree, _ = configs.circuit_3x3_d4()
    got, plan = run_gpu(net, tree)
    ref = _ref(net, tree)
    assert_close(got, ref, what="circuit_3x3_d4 vs oracle")
    net2, circ = grid_circuit_network(3, 3, 4, 0)
    sv = amplitudes(9, circ.gates, [])
    assert abs(complex(got) - complex(sv)) <= TOL_C64 * abs(complex(sv)) * 10


@pytest.mark.parametrize("n_open", [1, 3, 9])
def test_circuit_3x3_open_qubits(n_open):
    net, circ = grid_circuit_network(3, 3, 4, 0, n_open=n_open)
    tree = greedy_tree(net, 2)
    got, _ = run_gpu(net, tree)
    assert_close(got, _ref(net, tree), what=f"3x3 with {n_open} open")
    assert_close(got, amplitudes(9, circ.gates, list(range(n_open))), what="vs statevector")


def test_random_60_full():
    net, tree, _ = configs.random_60()
    got, plan = run_gpu(net, tree)
    assert_close(got, _ref(net, tree), what="random_60")


@pytest.mark.parametrize("seed", range(60))
def test_tiny_random_networks(seed):
    net = random_tiny_network(1000 + seed)
    tree = greedy_tree(net, seed, noise=0.5)
    got, _ = run_gpu(net, tree)
    assert_close(got, _ref(net, tree), what=f"tiny {seed}")


@pytest.mark.parametrize("seed", [2, 5])
def test_random_networks_mid(seed):
    net = random_network(40, seed)
    tree = greedy_tree(net, 0)
    got, _ = run_gpu(net, tree)
    assert_close(got, _ref(net, tree), what=f"random_40 seed {seed}")


def test_sliced_equals_oracle_and_unsliced():
    net = random_network(40, 2)
    tree = greedy_tree(net, 0)
    sl = choose_slices(net, tree, largest_intermediate(net, tree) // 8)[:3]
    assert len(sl) >= 1
    got_s, plan = run_gpu(net, tree, sl)
    assert plan.num_slices > 1
    got_u, _ = run_gpu(net, tree)
    ref = _ref(net, tree)
    assert_close(got_s, ref, what="sliced vs oracle")
    assert_close(got_s, got_u, what="sliced vs unsliced gpu")


def test_sliced_circuit_scalar():
    net, _ = grid_circuit_network(4, 4, 8, 3)
    tree = greedy_tree(net, 0)
    sl = choose_slices(net, tree, max(1, largest_intermediate(net, tree) // 16))[:4]
    got, plan = run_gpu(net, tree, sl)
    assert_close(got, _ref(net, tree), what="sliced 4x4 circuit")


def test_slice_shards_add_up():
    """tn_execute_slices: round-robin shards of the slices sum to the full
    result (the multi-GPU partition); an empty shard yields zeros."""
    import torch
    import exact_tensor_network_gb300 as tn
    net = random_network(40, 2)
    tree = greedy_tree(net, 0)
    sl = choose_slices(net, tree, largest_intermediate(net, tree) // 8)[:3]
    plan = tn.Plan.from_network(net, tree, sl)
    ns = plan.num_slices
    assert ns >= 4
    dev = torch.device("cuda:0")
    leaves = [torch.from_numpy(np.ascontiguousarray(d)).to(dev) for d in net.data]
    total = torch.zeros(plan.out_shape, dtype=torch.complex128, device=dev)
    for r in range(3):
        first, step, count = tn.shard_slices(ns, r, 3)
        o = torch.full(plan.out_shape, complex(5.0, 1.0), dtype=torch.complex64, device=dev)
        plan.execute_slices(leaves, o, first, step)
        total += o.to(torch.complex128)
    empty = torch.full(plan.out_shape, complex(5.0, 1.0), dtype=torch.complex64, device=dev)
    plan.execute_slices(leaves, empty, ns, 1)
    torch.cuda.synchronize()
    assert float(empty.abs().max()) == 0.0
    assert_close(total.cpu().numpy(), _ref(net, tree), what="sum of 3 slice shards")


@pytest.mark.parametrize("case", ["random_40", "circuit_4x4"])
def test_hoisting_matches_plain_slice_loop(case):
    """Slice-invariant hoisting (later slices rerun only the launches that
    depend on a sliced leaf) and the plain slice loop both match the oracle,
    over three replayed executes; hoisting launches less."""
    import torch
    import exact_tensor_network_gb300 as tn
    if case == "random_40":
        net = random_network(40, 2)
        tree = greedy_tree(net, 0)
        sl = choose_slices(net, tree, largest_intermediate(net, tree) // 8)[:3]
    else:
        net, _ = grid_circuit_network(4, 4, 8, 3)
        tree = greedy_tree(net, 0)
        sl = choose_slices(net, tree, max(1, largest_intermediate(net, tree) // 16))[:4]
    ref = _ref(net, tree)
    dev = torch.device("cuda:0")
    leaves = [torch.from_numpy(np.ascontiguousarray(d)).to(dev) for d in net.data]
    launches = {}
    for hoist in (True, False):
        plan = tn.Plan.from_network(net, tree, sl)
        plan.set_fusion(False)   # fused leaf subtrees would hold every launch here
        plan.set_hoisting(hoist)
        assert plan.num_slices > 1
        out = torch.full(plan.out_shape, complex(7.0, -3.0), dtype=torch.complex64, device=dev)
        for _ in range(3):
            plan.execute(leaves, out)
        torch.cuda.synchronize(dev)
        plan.check()
        launches[hoist] = plan.launches
        assert_close(out.cpu().numpy().astype(np.complex128), ref, what=f"{case} hoisting={hoist}")
    assert launches[True] < launches[False]


def test_repeated_execute_overwrites():
    net, tree, _ = configs.circuit_3x3_d4()
    got, _ = run_gpu(net, tree, repeat=3)
    assert_close(got, _ref(net, tree), what="three executes")


@pytest.mark.parametrize("lm,ln,lk", [(8, 8, 8), (0, 8, 8), (8, 0, 8), (8, 8, 0), (0, 0, 10),
                                      (9, 7, 5), (4, 12, 6)])
def test_single_node_shapes(lm, ln, lk):
    net = gemm_network(lm, ln, lk, lm * 100 + ln * 10 + lk)
    got, _ = run_gpu(net, [(0, 1)])
    assert_close(got, _ref(net, [(0, 1)]), what=f"gemm {lm},{ln},{lk}")


def test_single_leaf_permute_and_scalars():
    rng = np.random.default_rng(0)
    d = (rng.standard_normal((3, 5, 4, 2)) + 1j * rng.standard_normal((3, 5, 4, 2))).astype(np.complex64)
    net = Network([[0, 1, 2, 3]], [3, 5, 4, 2], [2, 0, 3, 1], [d])
    got, _ = run_gpu(net, [])
    assert_close(got, np.transpose(d, (2, 0, 3, 1)).astype(np.complex128), what="leaf permute")
    s = np.array(1.5 - 0.5j, dtype=np.complex64)
    v = (rng.standard_normal(7) + 0j).astype(np.complex64)
    net2 = Network([[], [0]], [7], [0], [s, v])
    got2, _ = run_gpu(net2, [(0, 1)])
    assert_close(got2, (s * v).astype(np.complex128), what="scalar leaf")


def test_extent_one_modes():
    rng = np.random.default_rng(3)
    ext = [1, 3, 1, 4, 2]
    tensors = [[0, 1, 2], [1, 3, 4], [2, 4, 0]]
    data = [(rng.standard_normal([ext[x] for x in t]) + 1j * rng.standard_normal([ext[x] for x in t]))
            .astype(np.complex64) for t in tensors]
    net = Network(tensors, ext, [3], data)
    tree = [(0, 1), (3, 2)]
    got, _ = run_gpu(net, tree)
    assert_close(got, _ref(net, tree), what="extent-1 modes")


def test_simt_policy_matches_auto():
    import exact_tensor_network_gb300 as tn
    net, tree, _ = configs.random_60()
    ref = _ref(net, tree)
    a, _ = run_gpu(net, tree, policy=tn.TN_POLICY_AUTO)
    b, _ = run_gpu(net, tree, policy=tn.TN_POLICY_SIMT)
    assert_close(a, ref, what="auto policy vs oracle")
    assert_close(b, ref, what="simt policy vs oracle")


@pytest.mark.parametrize("replay", [True, False])
def test_graph_replay_with_changing_buffers(replay):
    """Same buffers replay the recorded graph; new output or leaf buffers
    re-record; results match the oracle every time (and with replay off)."""
    import torch
    import exact_tensor_network_gb300 as tn
    net, tree, _ = configs.random_60()
    ref = _ref(net, tree)
    plan = tn.Plan.from_network(net, tree)
    tn.tn_plan_set_replay(plan.handle, replay)
    dev = torch.device("cuda:0")
    leaves = [torch.from_numpy(np.ascontiguousarray(d)).to(dev) for d in net.data]
    outs = [torch.zeros(plan.out_shape, dtype=torch.complex64, device=dev) for _ in range(2)]
    for it in range(6):
        o = outs[it // 3]
        o.fill_(complex(9.0, 9.0))
        if it == 4:
            leaves = [x.clone() for x in leaves]       # new leaf buffers
        plan.execute(leaves, o)
        torch.cuda.synchronize()
        assert_close(o.cpu().numpy().astype(np.complex128), ref, what=f"call {it}")
    plan.check()


def test_execute_inside_callers_graph_capture():
    """A caller capturing its stream records our launches in its graph."""
    import torch
    import exact_tensor_network_gb300 as tn
    net, tree, _ = configs.random_60()
    ref = _ref(net, tree)
    plan = tn.Plan.from_network(net, tree)
    dev = torch.device("cuda:0")
    leaves = [torch.from_numpy(np.ascontiguousarray(d)).to(dev) for d in net.data]
    out = torch.zeros(plan.out_shape, dtype=torch.complex64, device=dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        plan.execute(leaves, out, s)          # binds the workspace outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.execute(leaves, out, s)
    out.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy().astype(np.complex128), ref, what="caller graph replay")


@pytest.mark.parametrize("name", ["circuit_3x3_d4", "random_60"])
def test_tiny_batching_matches_unbatched(name):
    """Tiny nodes batched per schedule stage (auto) and launched one by one
    (no-tiny policy) both match the oracle."""
    import exact_tensor_network_gb300 as tn
    net, tree, _ = configs.by_name(name)
    ref = _ref(net, tree)
    a, pa = run_gpu(net, tree, policy=tn.TN_POLICY_AUTO, fuse=False)
    b, pb = run_gpu(net, tree, policy=tn.TN_POLICY_NO_TINY)
    assert pa.launches < pb.launches
    assert_close(a, ref, what=f"{name} batched tiny nodes")
    assert_close(b, ref, what=f"{name} one launch per node")


def _unitary_chain(pairs, seed):
    """Leaves 2i = U[a_i, x_i] and 2i + 1 = V[x_i, a_(i+1)], random 2 x 2
    unitaries (so every partial product stays unitary); a_0 and a_pairs are
    open.  The tree contracts every pair first (`pairs` tiny nodes in the
    first stage), then neighbours pairwise."""
    rng = np.random.default_rng(seed)
    tensors, data = [], []
    for i in range(pairs):
        tensors += [[i, pairs + 1 + i], [pairs + 1 + i, i + 1]]
    for _ in tensors:
        q, r = np.linalg.qr(rng.standard_normal((2, 2)) + 1j * rng.standard_normal((2, 2)))
        data.append((q * (np.diag(r) / np.abs(np.diag(r)))).astype(np.complex64))
    tree = [(2 * i, 2 * i + 1) for i in range(pairs)]
    cur, nid = [2 * pairs + i for i in range(pairs)], 3 * pairs
    while len(cur) > 1:
        nxt = []
        for x in range(0, len(cur) - 1, 2):
            tree.append((cur[x], cur[x + 1]))
            nxt.append(nid)
            nid += 1
        cur = nxt + ([cur[-1]] if len(cur) % 2 else [])
    return Network(tensors, [2] * (2 * pairs + 1), [0, pairs], data, f"chain_{pairs}"), tree


def test_tiny_stage_over_one_launch():
    """300 tiny nodes in one stage run as two batched launches (at most 256
    nodes each)."""
    import exact_tensor_network_gb300 as tn
    net, tree = _unitary_chain(300, 5)
    got, plan = run_gpu(net, tree, fuse=False)
    # 2 leaf launches (600 leaves, 512 per launch) + 10 tiny stages, the
    # first of them split in two
    assert plan.launches == 13
    ref = _ref(net, tree)
    assert_close(got, ref, what="300-node tiny stage")
    # a unitary, up to the complex64 rounding of 600 leaves
    assert np.allclose(ref @ ref.conj().T, np.eye(2), atol=1e-4)


def test_profiling_records_every_launch():
    import torch
    import exact_tensor_network_gb300 as tn
    net, tree, _ = configs.circuit_3x3_d4()
    plan = tn.Plan.from_network(net, tree)
    dev = torch.device("cuda:0")
    leaves = [torch.from_numpy(np.ascontiguousarray(d)).to(dev) for d in net.data]
    out = torch.empty(plan.out_shape, dtype=torch.complex64, device=dev)
    plan.set_profiling(True)
    plan.execute(leaves, out)
    torch.cuda.synchronize()
    recs = plan.profile()
    assert len(recs) == plan.launches
    assert all(r["ms"] >= 0 for r in recs)
    assert sum(r["flops"] for r in recs) == plan.flops


def _replay_case(case):
    import exact_tensor_network_gb300 as tn
    if case.startswith("random_60"):
        net, tree, _ = configs.random_60()
        pol = {"random_60_notiny": tn.TN_POLICY_NO_TINY, "random_60_simt": tn.TN_POLICY_SIMT}[case]
        return net, tree, [], pol
    if case == "circuit_3x3_sliced":
        net, tree, _ = configs.circuit_3x3_d4()
        return net, tree, net.closed_modes()[:3], tn.TN_POLICY_AUTO
    if case.startswith("tiny_sliced"):
        seed = int(case[-1])
        net = random_tiny_network(500 + seed)
        tree = greedy_tree(net, seed)
        sl = [x for x in net.closed_modes()][:2]
        return net, tree, sl, tn.TN_POLICY_NO_TINY if seed % 2 else tn.TN_POLICY_AUTO
    # a split-K tensor-core node (64 x 128 x 2048) feeding a split-K
    # streaming node (4 x 1 x 8192), two slices over the extra mode z
    rng = np.random.default_rng(41)
    ext = [64, 2048, 128, 4, 2]               # a x b e z
    tensors = [[0, 1, 4], [2, 1, 4], [3, 2, 0]]
    data = [((rng.standard_normal([ext[x] for x in t]) + 1j * rng.standard_normal([ext[x] for x in t]))
             * 0.05).astype(np.complex64) for t in tensors]
    net = Network(tensors, ext, [3], data)
    return net, [(0, 1), (3, 2)], [4], tn.TN_POLICY_AUTO


@pytest.mark.parametrize("case", ["random_60_notiny", "random_60_simt", "circuit_3x3_sliced",
                                  "tiny_sliced_0", "tiny_sliced_1", "splitk_sliced"])
def test_replayed_dependency_graph(case):
    """The recorded graph runs independent launches concurrently (ordered only
    where they touch common bytes); its replays match the oracle, including
    across slices (leaf buffers reused, the root adding into the output) and
    with split-K partials."""
    import torch
    import exact_tensor_network_gb300 as tn
    net, tree, sl, pol = _replay_case(case)
    ref = _ref(net, tree)
    plan = tn.Plan.from_network(net, tree, sl, "tf32x3", pol)
    if sl:
        assert plan.num_slices > 1
    dev = torch.device("cuda:0")
    leaves = [torch.from_numpy(np.ascontiguousarray(d)).to(dev) for d in net.data]
    out = torch.empty(plan.out_shape, dtype=torch.complex64, device=dev)
    for it in range(4):                        # direct, then three replays
        out.fill_(complex(9.0, -9.0))
        plan.execute(leaves, out)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy().astype(np.complex128), ref, what=f"{case} call {it}")
    plan.check()


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("case", ["random_60", "tiny_sliced"])
def test_execute_from_host_buffers(pinned, case):
    """tn_execute_host: host leaves in (pinned: one gather kernel over their
    device mappings; pageable: one copy each), contraction, result out."""
    import torch
    import exact_tensor_network_gb300 as tn
    if case == "random_60":
        net, tree, _ = configs.random_60()
        sl = []
    else:
        net = random_tiny_network(507)
        tree = greedy_tree(net, 7)
        sl = net.closed_modes()[:2]
    ref = _ref(net, tree)
    plan = tn.Plan.from_network(net, tree, sl)
    dev = torch.device("cuda:0")
    host_leaves = [torch.from_numpy(np.ascontiguousarray(d)) for d in net.data]
    host_out = torch.zeros(plan.out_shape, dtype=torch.complex64)
    if pinned:
        host_leaves = [h.pin_memory() for h in host_leaves]
        host_out = host_out.pin_memory()
    dev_leaves = [torch.empty_like(h, device=dev) for h in host_leaves]
    dev_out = torch.empty(plan.out_shape, dtype=torch.complex64, device=dev)
    for it in range(4):                        # direct, then recorded replays
        if it == 3:
            host_leaves[0].mul_(2.0)               # new values in the same buffer
            ref = 2.0 * ref                        # the result is linear in each leaf
        host_out.fill_(complex(5.0, 5.0))
        plan.execute_host(host_leaves, host_out, dev_leaves, dev_out)
        assert_close(host_out.numpy().astype(np.complex128), ref, what=f"{case} call {it}")
    call = plan.prepare_host(host_leaves, host_out, dev_leaves, dev_out)   # the prepared form
    for it in range(2):
        host_out.fill_(complex(5.0, 5.0))
        call()
        assert_close(host_out.numpy().astype(np.complex128), ref, what=f"{case} prepared call {it}")
    plan.check()


# ---- TN_PREC_FP32: every node on CUDA-core fp32 FMA ------------------------

@pytest.mark.parametrize("case", ["circuit_3x3_d4", "random_60", "sliced_30", "twin_4x4_d12"])
def test_fp32_precision_networks(case):
    """The fp32 precision against the oracle at the complex64 tolerance:
    no node may reach the tensor cores."""
    from helpers import TOL_C64
    sl = []
    if case == "circuit_3x3_d4":
        net, tree, _ = configs.circuit_3x3_d4()
    elif case == "random_60":
        net, tree, _ = configs.random_60()
    elif case == "sliced_30":
        net = random_network(30, 4)
        tree = greedy_tree(net, 0)
        sl = choose_slices(net, tree, largest_intermediate(net, tree) // 8)[:3]
    else:
        net, _ = grid_circuit_network(4, 4, 12, 2, n_open=6)
        tree = greedy_tree(net, 28, noise=0.6, alpha=0.25)
    got, plan = run_gpu(net, tree, sl, precision="fp32")
    assert all(plan.node_class(s) != 1 for s in range(len(tree)))
    if sl:
        assert plan.num_slices > 1
    assert_close(got, _ref(net, tree, sl), TOL_C64, f"{case} fp32")


@pytest.mark.parametrize("m,n,k", [(512, 512, 512), (300, 257, 1000), (1, 1, 4096), (4096, 3, 16),
                                   (64, 2048, 2), (129, 65, 1)])
def test_fp32_precision_nodes(m, n, k):
    from helpers import TOL_C64, node_network
    net = node_network(m, n, k, m * 7 + n * 3 + k)
    got, plan = run_gpu(net, [(0, 1)], precision="fp32", policy=2)
    assert plan.node_class(0) != 1
    assert_close(got, _ref(net, [(0, 1)]), TOL_C64, f"fp32 node {m}x{n}x{k}")


def test_reduced_precision_errors_reported():
    """Reported, not gated (the bf16 tolerance is gated on single nodes):
    max |gpu - ref| / max |ref| of every precision on the 3x3 circuit, the
    random 60-tensor network and the 4x4 x 12-cycle twin of the 6x6 recipe.
    Only a loose sanity bound applies here."""
    from helpers import max_rel_err
    cases = {"circuit_3x3_d4": configs.circuit_3x3_d4()[:2], "random_60": configs.random_60()[:2]}
    net, _ = grid_circuit_network(4, 4, 12, 2, n_open=6)
    cases["twin_4x4_d12"] = (net, greedy_tree(net, 28, noise=0.6, alpha=0.25))
    for name, (net, tree) in cases.items():
        ref = _ref(net, tree)
        line = []
        for prec in ("tf32x3", "bf16x3", "bf16", "fp32"):
            got, _ = run_gpu(net, tree, precision=prec)
            r = max_rel_err(got, ref)
            line.append(f"{prec} {r:.2e}")
            assert np.isfinite(r) and r < 0.5, f"{name} {prec}: {r}"
        print(f"precision errors {name}: " + ", ".join(line))


# ---- leaf permutation paths: conversions and true transposes ----------------

@pytest.mark.parametrize("perm,shape,policy", [
    ((1, 0), (96, 200), 2),         # a transpose into a CUDA-core operand
    ((1, 0), (300, 256), 2),
    ((2, 0, 1), (40, 64, 48), 2),   # contiguous axis in the middle of the destination
    ((1, 0), (256, 2048), 0),       # a transpose into a K-tiled tensor-core operand
    ((0, 1), (4096, 2048), 0),      # a pure conversion (K-tiled split tf32)
    ((0, 1), (256, 1000), 0),       # a pure conversion, untiled, ragged k
])
def test_leaf_permutation_paths(perm, shape, policy):
    """Leaf A[i, x] (possibly several i modes) stored in a permuted order,
    contracted with B[j, x]: the leaf permutation moves it into lifetime
    order (and the tensor-core operand format) through the shared-memory
    transpose, the contiguous conversion or the general path."""
    rng = np.random.default_rng(sum(shape))
    modes_a = list(range(len(shape)))          # A's modes in lifetime order: [M..., x]
    x = len(shape) - 1
    ext = list(shape) + [64]                    # last extra mode: j (B's kept mode)
    j = len(shape)
    stored = [modes_a[p] for p in perm]         # user order of A
    a = (rng.standard_normal([ext[m] for m in stored]) +
         1j * rng.standard_normal([ext[m] for m in stored])).astype(np.complex64)
    b = (rng.standard_normal((ext[j], ext[x])) + 1j * rng.standard_normal((ext[j], ext[x]))).astype(np.complex64)
    open_modes = modes_a[:-1] + [j]
    net = Network([stored, [j, x]], ext, open_modes, [a, b], f"perm_{perm}_{shape}")
    got, plan = run_gpu(net, [(0, 1)], policy=policy)
    assert_close(got, _ref(net, [(0, 1)]), what=f"leaf {perm} {shape}")
