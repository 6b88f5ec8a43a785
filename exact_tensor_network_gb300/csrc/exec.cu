// Executor: node classification and the stream-ordered launch sequence.
//
// For every slice (section 1.1 of "Crossing the single-GPU memory wall":
// the sliced sub-contractions are independent and their results add up) the
// executor permutes the leaves that need it, then runs the tree's steps in
// order, each on the kernel its class selects; the root step writes the
// caller's output on the first slice and adds into it on later ones.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <string>

#include "kernels.h"
#include "plan.h"

namespace tn {

// Node classes.  A node goes to the tensor cores when its operands can be
// TMA-tiled (k entries per row a multiple of 16 bytes in the planar
// format), its tiles are reasonably full (m, n >= 64, k >= 16), and its
// arithmetic intensity with planar operand bytes (16 per tf32x3 entry,
// 4 per bf16 entry, 8 per output entry) is high enough to be
// compute-bound rather than bandwidth-bound.
int classify(const Plan &p, const NodePlan &nd) {
    if (p.policy == TN_POLICY_SIMT) return TN_NODE_SIMT;
    const bool bf16 = p.precision == TN_PREC_BF16;
    const bool bf16x3 = p.precision == TN_PREC_BF16X3;
    const bool fp32 = p.precision == TN_PREC_FP32;
    const uint64_t kq = bf16 || bf16x3 ? 8 : 4;   // 16-byte rows of a TMA box
    if (p.policy == kPolicyForceDense)
        return (!fp32 && nd.k % kq == 0) ? TN_NODE_DENSE : TN_NODE_SIMT;
    if (p.policy == TN_POLICY_AUTO && nd.m * nd.n * nd.k <= kTinyMacs && nd.k <= kTinyMaxK &&
        nd.m * nd.n <= kTinyMaxOut)
        return TN_NODE_TINY;
    if (!fp32 && nd.k % kq == 0 && nd.k >= 16 && nd.m >= 64 && nd.n >= 64) {
        const double in_b = bf16 ? 4.0 : bf16x3 ? 8.0 : 16.0;
        const double m = (double)nd.m, n = (double)nd.n, k = (double)nd.k;
        const double intensity = 8.0 * m * n * k / (in_b * (m * k + n * k) + 8.0 * m * n);
        if (intensity >= 24.0) return TN_NODE_DENSE;
    }
    if (std::min(nd.m, nd.n) <= (uint64_t)kStreamMaxN) return TN_NODE_STREAM;
    return TN_NODE_SIMT;
}

namespace {

// Stream-kernel shape: threads per row of A and rows per CTA.
void stream_shape(uint64_t rows, uint64_t k, int *lanes, int64_t *rows_per_cta) {
    int l = 1;
    while (l < 32 && (uint64_t)l * 8 < k) l *= 2;
    const int64_t groups = 256 / l;
    int64_t mult = (int64_t)(rows / ((uint64_t)groups * 4 * kTargetCtas));
    if (mult < 1) mult = 1;
    *lanes = l;
    *rows_per_cta = groups * mult;
}

constexpr uint64_t kPartialBudget = 1ull << 30;   // bytes of split-K partials per node

}  // namespace

// Split-K for the CUDA-core classes: cut k when the node alone would not
// give every SM two CTAs, keeping chunks of at least 64 entries.
void choose_split(const Plan &p, NodePlan &nd) {
    nd.ksplit = 1;
    nd.kchunk = (int64_t)nd.k;
    nd.swap = 0;
    nd.narrow = 0;
    nd.pair = 0;
    nd.tail_first = -1;
    nd.red_ctas = 0;
    uint64_t units = 0, outs = nd.m * nd.n;
    if (nd.cls == TN_NODE_DENSE) {
        // a side of at most 64 goes to N (operands swapped when it is m) and
        // the node runs 128 x 64 tiles
        if (std::min(nd.m, nd.n) <= (uint64_t)(kDenseBN / 2)) {
            nd.swap = nd.m < nd.n ? 1 : 0;
            nd.narrow = 1;
        } else if (nd.k < 512 && 2 * ((nd.m + kDenseBM - 1) / kDenseBM) * ((nd.n + kDenseBN - 1) / kDenseBN) <=
                                     (uint64_t)(kTargetCtas / 2)) {
            // a short-k node whose 128 x 128 tiles would fill at most half
            // the SMs: its time is the epilogue, which 128 x 64 tiles spread
            // over twice the CTAs (512 x 2048 x 32: 22.7 -> 17.3 us)
            nd.narrow = 1;
        } else if (p.cta_pairs && std::max(nd.m, nd.n) >= (uint64_t)(2 * kDenseBM)) {
            // CTA pairs: tiles of 256 rows (the longer side) x 128 columns
            nd.swap = nd.m < 2 * (uint64_t)kDenseBM ? 1 : 0;
            nd.pair = 1;
        }
        // tensor-core tiles are 128 x 128 (or 128 x 64; pairs 256 x 128 on
        // two SMs) and one CTA runs per SM; splits are whole multiples of the
        // 256-entry k chunk
        const uint64_t tiles = dense_tiles(nd);
        const uint64_t sms = nd.pair ? kTargetCtas / 4 : kTargetCtas / 2;
        if (tiles >= sms) {
            if (nd.narrow || nd.pair) return;   // no tail split on narrow tiles or pairs
            // a last wave at most half full runs its tiles as two k halves:
            // it then takes half a tile's time instead of a whole one
            const uint64_t tail = tiles % sms;
            if (tail > 0 && 2 * tail <= sms && nd.k >= 512) nd.tail_first = (int64_t)(tiles - tail);
            return;
        }
        if (nd.k < 512) return;
        // the split count whose tiles x splits work items fill their waves
        // best (fewer splits when nearly equal: each split adds partials to
        // write and reduce); splits are whole 256-entry chunks
        const uint64_t smax = std::min<uint64_t>(std::min<uint64_t>(nd.k / 256, 64),
                                                 kPartialBudget / (8 * outs));
        uint64_t s = 1;
        double best = (double)tiles / (double)sms;
        for (uint64_t c = 2; c <= smax; ++c) {
            const uint64_t items = tiles * c, waves = (items + sms - 1) / sms;
            const double eff = (double)items / (double)(waves * sms);
            if (eff > best + 0.02) {
                best = eff;
                s = c;
            }
        }
        if (s < 2) return;
        uint64_t chunk = (nd.k + s - 1) / s;
        chunk = (chunk + 255) / 256 * 256;
        const uint64_t ks = (nd.k + chunk - 1) / chunk;
        if (ks < 2) return;
        nd.kchunk = (int64_t)chunk;
        nd.ksplit = (int32_t)ks;
        return;
    }
    if (nd.cls == TN_NODE_STREAM) {
        nd.swap = nd.m < nd.n ? 1 : 0;
        const uint64_t rows = std::max(nd.m, nd.n);
        int lanes;
        int64_t rpc;
        stream_shape(rows, nd.k, &lanes, &rpc);
        units = (rows + rpc - 1) / rpc;
        nd.red_ctas = (int64_t)units;
    } else if (nd.cls == TN_NODE_SIMT) {
        units = ((nd.m + 63) / 64) * ((nd.n + 63) / 64);
    } else {
        return;
    }
    if (units >= (uint64_t)kTargetCtas || nd.k < 128) return;
    uint64_t s = std::min<uint64_t>((kTargetCtas + units - 1) / units, nd.k / 64);
    s = std::min<uint64_t>(s, kPartialBudget / (8 * outs));
    s = std::min<uint64_t>(s, 4096);
    if (s < 2) return;
    uint64_t chunk = (nd.k + s - 1) / s;
    chunk = (chunk + 15) / 16 * 16;
    nd.kchunk = (int64_t)chunk;
    nd.ksplit = (int32_t)((nd.k + chunk - 1) / chunk);
    if (nd.ksplit < 2) {
        nd.ksplit = 1;
        nd.kchunk = (int64_t)nd.k;
    }
}

// Split-K nodes of the streaming class reduce their partials in the node
// kernel (the last split to finish a row block); the others get a reduction
// launch, which spreads the sums over every SM (the tensor-core kernel's
// last splits alone took longer than kernel plus reduction).
bool fused_reduction(const NodePlan &nd) { return nd.cls == TN_NODE_STREAM && nd.ksplit > 1; }

// The program a slice runs: the whole schedule (the first slice of an
// execute, or every slice without hoisting) or the variant launches only.
struct Program {
    const std::vector<Launch> &sched;
    const std::vector<int32_t> &jobs;     // perm_table entries
    const std::vector<int32_t> &groups;   // fused groups (LAUNCH_FUSED ranges index this)
};
Program program(const Plan &p, bool first) {
    if (first || !(p.hoist && p.n_slices > 1)) return {p.sched, p.perm_all, p.fuse_all};
    return {p.sched_rest, p.perm_rest, p.fuse_rest};
}

uint64_t launches_of(const Plan &p, bool first) {
    const Program g = program(p, first);
    uint64_t n = (g.jobs.size() + kPermBatch - 1) / kPermBatch;
    for (const auto &L : g.sched) {
        if (L.kind == LAUNCH_TINY || L.kind == LAUNCH_FUSED) ++n;
        if (L.kind == LAUNCH_NODE) n += fused_reduction(p.nodes[L.node]) ? 1 : p.nodes[L.node].ksplit > 1 ? 2 : 1;
    }
    return n;
}

void drop_graph(Plan *p) {
    if (p->graph_exec) cudaGraphExecDestroy(static_cast<cudaGraphExec_t>(p->graph_exec));
    p->graph_exec = nullptr;
    if (p->host_graph_exec) cudaGraphExecDestroy(static_cast<cudaGraphExec_t>(p->host_graph_exec));
    p->host_graph_exec = nullptr;
    p->hg_key.clear();
    p->graph_leaves.clear();
    p->graph_out = nullptr;
    p->graph_ws = nullptr;
}

void release_events(Plan *p) {
    for (void *e : p->events)
        if (e) cudaEventDestroy(static_cast<cudaEvent_t>(e));
    p->events.clear();
    for (void *e : p->dag_events)
        if (e) cudaEventDestroy(static_cast<cudaEvent_t>(e));
    p->dag_events.clear();
    drop_graph(p);
    if (p->capture_stream) cudaStreamDestroy(static_cast<cudaStream_t>(p->capture_stream));
    p->capture_stream = nullptr;
    for (void *s : p->lane_streams)
        if (s) cudaStreamDestroy(static_cast<cudaStream_t>(s));
    p->lane_streams.clear();
}

namespace {

// Brackets launches with CUDA events when the plan is being profiled.
struct Recorder {
    Plan *p;
    cudaStream_t s;
    size_t i = 0;
    bool ok = true;
    void begin(int32_t kernel, int32_t step, uint64_t flops, uint64_t bytes) {
        if (!p->profiling || !ok) return;
        while (p->events.size() < 2 * (i + 1)) {
            cudaEvent_t e;
            if (cudaEventCreate(&e) != cudaSuccess) {
                ok = false;
                return;
            }
            p->events.push_back(e);
        }
        cudaEventRecord(static_cast<cudaEvent_t>(p->events[2 * i]), s);
        p->records.push_back(tn_launch_record{kernel, step, 0.f, flops, bytes});
    }
    void end() {
        if (!p->profiling || !ok) return;
        cudaEventRecord(static_cast<cudaEvent_t>(p->events[2 * i + 1]), s);
        ++i;
    }
};

tn_status cuda_fail(Plan *p, cudaError_t e, const char *what);

// ---- dependency graph of the launches, for recording ----
//
// What each launch reads and writes: byte ranges of the workspace arena, or
// the caller's output (one token: lo < 0).  Leaves read in place are never
// written and are left out.  Two launches conflict when one writes what the
// other reads or writes; every order that keeps conflicting launches in
// their issue order computes the same result as the issue order itself.
struct Range {
    int64_t lo, hi;
};
struct Access {
    std::vector<Range> rd, wr;
};

void add_range(std::vector<Range> &v, const Place &pl, uint64_t bytes) {
    if (pl.kind == PLACE_WS) v.push_back({(int64_t)pl.off, (int64_t)(pl.off + bytes)});
    else if (pl.kind == PLACE_OUT) v.push_back({-1, -1});
}

bool overlap(const std::vector<Range> &x, const std::vector<Range> &y) {
    for (const Range &a : x)
        for (const Range &b : y) {
            if (a.lo < 0 || b.lo < 0) {
                if (a.lo < 0 && b.lo < 0) return true;
                continue;
            }
            if (a.lo < b.hi && b.lo < a.hi) return true;
        }
    return false;
}

bool conflict(const Access &e, const Access &l) {
    return overlap(e.wr, l.rd) || overlap(e.wr, l.wr) || overlap(e.rd, l.wr);
}

// Accesses of one slice's launches (the first slice's program or a later
// one's), in the order execute_range issues them.
std::vector<Access> slice_accesses(const Plan &p, bool first) {
    const Program g = program(p, first);
    std::vector<Access> acc;
    const int njobs = (int)g.jobs.size();
    for (int j0 = 0; j0 < njobs; j0 += kPermBatch) {
        Access a;
        for (int j = j0; j < std::min(njobs, j0 + kPermBatch); ++j) {
            const PermDesc &d = p.perm_table[g.jobs[j]];
            if (d.dst_off < 0) a.wr.push_back({-1, -1});
            else a.wr.push_back({d.dst_off, d.dst_off + d.size * (int64_t)fmt_bytes(d.fmt)});
        }
        acc.push_back(a);
    }
    const TinyDesc *tiny = reinterpret_cast<const TinyDesc *>(
        p.table_blob.data() + (p.tiny_off - p.table_off));
    for (const Launch &L : g.sched) {
        if (L.kind == LAUNCH_PERMUTE) continue;
        if (L.kind == LAUNCH_FUSED) {
            // reads only the caller's leaves; writes the groups' roots
            Access a;
            for (int x = L.first; x < L.first + L.count; ++x) {
                const NodePlan &rn = p.nodes[p.fuse_groups[g.groups[x]].step];
                add_range(a.wr, rn.pc, rn.m * rn.n * fmt_bytes(rn.out_fmt));
            }
            acc.push_back(a);
            continue;
        }
        if (L.kind == LAUNCH_TINY) {
            Access a;
            for (int i = L.first; i < L.first + L.count; ++i) {
                const TinyDesc &d = tiny[i];
                const int64_t m = d.m, n = d.n, k = d.k;
                a.rd.push_back({d.a_off, d.a_off + 8 * m * k});
                a.rd.push_back({d.b_off, d.b_off + 8 * n * k});
                if (d.c_off < 0) a.wr.push_back({-1, -1});
                else a.wr.push_back({d.c_off, d.c_off + m * n * (int64_t)fmt_bytes(d.out_fmt)});
            }
            acc.push_back(a);
            continue;
        }
        const NodePlan &nd = p.nodes[L.node];
        Access a;
        add_range(a.rd, nd.pa, nd.m * nd.k * fmt_bytes(p.fmt[nd.a]));
        add_range(a.rd, nd.pb, nd.n * nd.k * fmt_bytes(p.fmt[nd.b]));
        add_range(a.wr, nd.pc, nd.m * nd.n * fmt_bytes(nd.out_fmt));
        if (nd.tail_first >= 0) add_range(a.wr, nd.part, part_bytes(nd));
        if (nd.ksplit > 1 && fused_reduction(nd)) {
            add_range(a.wr, nd.part, part_bytes(nd));
            acc.push_back(a);
        } else if (nd.ksplit > 1) {
            add_range(a.wr, nd.part, part_bytes(nd));
            acc.push_back(a);
            Access r;
            add_range(r.rd, nd.part, part_bytes(nd));
            add_range(r.wr, nd.pc, nd.m * nd.n * fmt_bytes(nd.out_fmt));
            acc.push_back(r);
        } else {
            acc.push_back(a);
        }
    }
    return acc;
}

constexpr int kLanes = 6;   // streams a recording spreads independent launches over

// Issues the launches of a recording on several streams: launch i waits
// (by event) for the launches it conflicts with on other streams and
// follows the previous launch of its own stream.  Stream 0 is the capture
// stream; the others join the capture through those waits and are joined
// back into stream 0 at the end.
struct Dag {
    std::vector<cudaStream_t> lane_stream;
    std::vector<cudaEvent_t> ev;
    std::vector<int> lane;                    // per launch
    std::vector<std::vector<int>> wait;       // per launch: launches to wait for
    std::vector<int> tail;                    // per stream: last launch
    size_t next = 0;
    bool ok = true;

    cudaStream_t begin() {
        const size_t i = next;
        cudaStream_t s = lane_stream[lane[i]];
        for (int e : wait[i])
            if (cudaStreamWaitEvent(s, ev[e], 0) != cudaSuccess) ok = false;
        return s;
    }
    void end() {
        const size_t i = next++;
        if (cudaEventRecord(ev[i], lane_stream[lane[i]]) != cudaSuccess) ok = false;
    }
    bool join() {
        for (size_t l = 1; l < lane_stream.size(); ++l)
            if (tail[l] >= 0 && cudaStreamWaitEvent(lane_stream[0], ev[tail[l]], 0) != cudaSuccess)
                return false;
        return ok;
    }
};

// Dependencies and streams of all launches of slices first, first + step, ...
tn_status build_dag(Plan *p, cudaStream_t origin, uint64_t first, uint64_t step, Dag *d) {
    // every launch of the range in issue order: the first slice's program,
    // then the later slices'
    std::vector<Access> all;
    if (first < p->n_slices) {
        all = slice_accesses(*p, true);
        const std::vector<Access> later = slice_accesses(*p, false);
        for (uint64_t s = first + step; s < p->n_slices; s += step)
            all.insert(all.end(), later.begin(), later.end());
    }
    const size_t N = all.size();
    while (p->lane_streams.size() < (size_t)kLanes - 1) {
        cudaStream_t s;
        cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
        if (e != cudaSuccess) return cuda_fail(p, e, "creating a stream");
        p->lane_streams.push_back(s);
    }
    while (p->dag_events.size() < N) {
        cudaEvent_t ev;
        cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(p, e, "creating an event");
        p->dag_events.push_back(ev);
    }
    d->lane_stream.assign(1, origin);
    for (void *s : p->lane_streams) d->lane_stream.push_back(static_cast<cudaStream_t>(s));
    d->ev.resize(N);
    for (size_t i = 0; i < N; ++i) d->ev[i] = static_cast<cudaEvent_t>(p->dag_events[i]);
    d->lane.assign(N, 0);
    d->wait.assign(N, {});
    d->tail.assign(kLanes, -1);
    d->next = 0;
    std::vector<int> last(kLanes);
    for (size_t i = 0; i < N; ++i) {
        // latest conflicting launch on each stream
        std::fill(last.begin(), last.end(), -1);
        bool any = false;
        for (size_t e = 0; e < i; ++e)
            if (conflict(all[e], all[i])) {
                last[d->lane[e]] = std::max(last[d->lane[e]], (int)e);
                any = true;
            }
        // a stream whose last launch is one of those adds no false order;
        // else an unused stream; else the stream with the oldest last launch
        int l = -1;
        if (!any) {
            l = 0;   // joins nothing: stays on the capture stream
        } else {
            for (int c = 0; c < kLanes; ++c)
                if (d->tail[c] >= 0 && last[c] == d->tail[c] && (l < 0 || d->tail[c] > d->tail[l])) l = c;
            if (l < 0)
                for (int c = 1; c < kLanes && l < 0; ++c)
                    if (d->tail[c] < 0) l = c;
            if (l < 0) {
                l = 0;
                for (int c = 1; c < kLanes; ++c)
                    if (d->tail[c] < d->tail[l]) l = c;
            }
        }
        d->lane[i] = l;
        for (int c = 0; c < kLanes; ++c)
            if (c != l && last[c] >= 0) d->wait[i].push_back(last[c]);
        d->tail[l] = (int)i;
    }
    return TN_OK;
}

uint64_t node_bytes(const NodePlan &nd, bool accumulate) {
    return 8 * (nd.m * nd.k + nd.n * nd.k + nd.m * nd.n * (accumulate ? 2 : 1));
}

tn_status cuda_fail(Plan *p, cudaError_t e, const char *what) {
    p->last_error = std::string(what) + ": " + cudaGetErrorString(e);
    return TN_ECUDA;
}

// TMA maps of every tensor-core node's planar operands inside the current
// workspace (host-side encoding only; rebuilt when the workspace moves).
tn_status build_dense_maps(Plan *p) {
    p->dense_maps.clear();
    char *arena = static_cast<char *>(p->ws) + p->arena_off;
    for (size_t s = 0; s < p->nodes.size(); ++s) {
        const NodePlan &nd = p->nodes[s];
        if (nd.cls != TN_NODE_DENSE) continue;
        if (nd.pa.kind != PLACE_WS || nd.pb.kind != PLACE_WS) {
            p->last_error = "tensor-core operand not in the workspace";
            return TN_EDEVICE;
        }
        DenseMaps dm;
        std::memset(&dm, 0, sizeof(dm));
        dm.node = (int32_t)s;
        std::string err;
        // kernel view: A = the operand with the rows, B = the one with the
        // columns (swapped when the node runs C^T = B A^T)
        const Place &pa = nd.swap ? nd.pb : nd.pa, &pb = nd.swap ? nd.pa : nd.pb;
        const int32_t fa = p->fmt[nd.swap ? nd.b : nd.a], fb = p->fmt[nd.swap ? nd.a : nd.b];
        const int32_t brows = (nd.narrow || nd.pair) ? (int32_t)(kDenseBN / 2) : (int32_t)kDenseBN;
        if (!encode_operand_map(&dm.a, arena + pa.off, (int64_t)dense_rows(nd), (int64_t)nd.k, fa,
                                nd.ktiled != 0, (int32_t)kDenseBM, &err) ||
            !encode_operand_map(&dm.b, arena + pb.off, (int64_t)dense_cols(nd), (int64_t)nd.k, fb,
                                nd.ktiled != 0, brows, &err)) {
            p->last_error = "step " + std::to_string(s) + ": " + err;
            return TN_ECUDA;
        }
        p->dense_maps.push_back(dm);
    }
    p->maps_ws = p->ws;
    return TN_OK;
}

}  // namespace

tn_status upload_tables(Plan *p) {
    cudaError_t e = cudaMemset(p->ws, 0, p->table_off);
    if (e != cudaSuccess) return cuda_fail(p, e, "clearing the status word");
    if (!p->table_blob.empty()) {
        e = cudaMemcpy(static_cast<char *>(p->ws) + p->table_off, p->table_blob.data(),
                       p->table_blob.size(), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(p, e, "uploading the descriptor tables");
    }
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(p, e, "querying the SM count");
    return build_dense_maps(p);
}

// Slices first, first + step, ... of the plan; the first of them writes the
// output and the others add into it; an empty range zeroes the output.
namespace {

// Slices first, first + step, ... issued on `stream`, or, with a graph
// recorder, each launch on the stream the recorder picks for it.
// With stop_launch >= 0, only the first slice's program runs, and only up to
// and including its launch of that index in sched (tn_execute_prefix).
tn_status issue_range(Plan *p, const void *const *leaf_ptrs, void *out_ptr, cudaStream_t stream,
                      uint64_t first, uint64_t step, Dag *dag, int32_t stop_launch = -1) {
    if (first >= p->n_slices) {
        cudaError_t e = cudaMemsetAsync(out_ptr, 0, p->out_elems * sizeof(float2), stream);
        return e == cudaSuccess ? TN_OK : cuda_fail(p, e, "zeroing the output");
    }
    if (stop_launch < 0) p->prefix_step = -1;   // the buffers are about to be reused
    char *ws = static_cast<char *>(p->ws);
    char *arena = ws + p->arena_off;
    DevStatus *status = reinterpret_cast<DevStatus *>(ws);
    const PermDesc *table = reinterpret_cast<const PermDesc *>(ws + p->table_off);
    float2 *out = static_cast<float2 *>(out_ptr);
    const int n = p->n_tensors;
    const int nsl = (int)p->slice_modes.size();
    std::vector<int64_t> digit(nsl, 0);
    std::vector<const float2 *> leaf_src(n);
    tn_status st = TN_OK;
    if (p->maps_ws != p->ws) {
        st = build_dense_maps(p);
        if (st != TN_OK) return st;
    }
    if (p->num_sms <= 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(p, e, "querying the SM count");
    }
    std::vector<int32_t> map_of(p->nodes.size(), -1);
    for (size_t i = 0; i < p->dense_maps.size(); ++i) map_of[p->dense_maps[i].node] = (int32_t)i;
    PermLaunch *pl = new PermLaunch;
    Recorder rec{p, stream};
    if (p->profiling) p->records.clear();   // records of an earlier profiled run stay otherwise

    for (uint64_t sigma = first; sigma < p->n_slices && st == TN_OK; sigma += step) {
        const bool later = sigma != first;   // add into the output
        const Program g = program(*p, !later);
        // slice digits, first slice mode most significant
        uint64_t rem = sigma;
        for (int i = nsl - 1; i >= 0; --i) {
            digit[i] = (int64_t)(rem % (uint64_t)p->slice_ext[i]);
            rem /= (uint64_t)p->slice_ext[i];
        }
        for (int t = 0; t < n; ++t) {
            int64_t off = 0;
            for (const auto &term : p->leaves[t].slice_terms) off += digit[term.first] * term.second;
            leaf_src[t] = static_cast<const float2 *>(leaf_ptrs[t]) + off;
        }
        // leaf permutations, batched
        const int njobs = (int)g.jobs.size();
        for (int j0 = 0; j0 < njobs; j0 += kPermBatch) {
            const int cnt = std::min(kPermBatch, njobs - j0);
            pl->njobs = cnt;
            pl->accumulate = 0;
            pl->table = table;
            pl->arena = arena;
            pl->out = out;
            int ctas = 0;
            for (int j = 0; j < cnt; ++j) {
                const int32_t job = g.jobs[j0 + j];
                pl->job[j] = job;
                pl->cta_start[j] = ctas;
                pl->src[j] = leaf_src[p->perm_leaves[job]];
                ctas += permute_job_ctas(p->perm_table[job]);
            }
            pl->cta_start[cnt] = ctas;
            // algorithmic bytes: every entry read once (complex64) and written
            // once in the destination's format
            uint64_t bytes = 0;
            for (int j = 0; j < cnt; ++j) {
                const PermDesc &pd = p->perm_table[g.jobs[j0 + j]];
                bytes += (8 + fmt_bytes(pd.dst_off < 0 ? (int32_t)FMT_C64 : pd.fmt)) * (uint64_t)pd.size;
            }
            rec.begin(TN_KERNEL_PERMUTE, -1, 0, bytes);
            cudaError_t e = launch_permute(*pl, ctas, dag ? dag->begin() : stream);
            if (dag) dag->end();
            rec.end();
            if (e != cudaSuccess) {
                st = cuda_fail(p, e, "launching the leaf permutation");
                break;
            }
        }
        if (st != TN_OK) break;
        if (stop_launch >= 0) p->prefix_leaves.assign(leaf_src.begin(), leaf_src.end());
        for (size_t li = 0; li < g.sched.size(); ++li) {
            const Launch &L = g.sched[li];
            if (stop_launch >= 0 && (int32_t)li > stop_launch) break;
            if (L.kind == LAUNCH_PERMUTE) continue;   // issued above
            if (L.kind == LAUNCH_FUSED) {
                FuseLaunch *fl = new FuseLaunch;
                std::memset(fl, 0, sizeof(FuseLaunch));
                fl->ngroups = L.count;
                fl->accumulate_root = later ? 1 : 0;
                fl->groups = reinterpret_cast<const FuseGroup *>(ws + p->fuse_off);
                fl->nodes = reinterpret_cast<const FuseNode *>(ws + p->fuse_node_off);
                fl->gather = reinterpret_cast<const FuseGather *>(ws + p->fuse_gather_off);
                fl->levels = reinterpret_cast<const int32_t *>(ws + p->fuse_lvl_off);
                fl->offs = reinterpret_cast<const int32_t *>(ws + p->fuse_offs_off);
                fl->chunks = reinterpret_cast<const int32_t *>(ws + p->fuse_chunk_off);
                fl->arena = arena;
                fl->out = out;
                int nsrc = 0, smem = 0;
                for (int x = 0; x < L.count; ++x) {
                    const int32_t gi = g.groups[L.first + x];
                    const FuseGroup &G = p->fuse_groups[gi];
                    fl->group[x] = gi;
                    fl->src_first[x] = nsrc;
                    for (int l = 0; l < G.n_leaves; ++l)
                        fl->src[nsrc++] = leaf_src[p->fuse_leaves_host[G.first_leaf + l].leaf];
                    smem = std::max(smem, G.smem_bytes);
                }
                rec.begin(TN_KERNEL_FUSED, -1, L.flops, L.bytes);
                cudaError_t e = launch_fused(*fl, smem, dag ? dag->begin() : stream);
                if (dag) dag->end();
                rec.end();
                delete fl;
                if (e != cudaSuccess) {
                    st = cuda_fail(p, e, "launching the fused leaf subtrees");
                    break;
                }
                continue;
            }
            if (L.kind == LAUNCH_TINY) {
                TinyLaunch tl;
                tl.table = reinterpret_cast<const TinyDesc *>(ws + p->tiny_off);
                tl.first = L.first;
                tl.count = L.count;
                tl.arena = arena;
                tl.out = out;
                tl.accumulate_root = later ? 1 : 0;
                const unsigned char *descs = p->table_blob.data() + (p->tiny_off - p->table_off);
                for (int x = 0; x < L.count; ++x) {
                    TinyDesc d;
                    std::memcpy(&d, descs + (size_t)(L.first + x) * sizeof(TinyDesc), sizeof(d));
                    tl.base[x] = d.cta_base;
                }
                tl.base[L.count] = L.ctas;
                rec.begin(TN_KERNEL_TINY, -1, L.flops, L.bytes);
                cudaError_t e = launch_tiny_batch(tl, L.ctas, dag ? dag->begin() : stream);
                if (dag) dag->end();
                rec.end();
                if (e != cudaSuccess) {
                    st = cuda_fail(p, e, "launching a tiny-node batch");
                    break;
                }
                continue;
            }
            const NodePlan &nd = p->nodes[L.node];
            auto resolve = [&](const Place &pl_) -> float2 * {
                switch (pl_.kind) {
                    case PLACE_WS: return reinterpret_cast<float2 *>(arena + pl_.off);
                    case PLACE_LEAF: return const_cast<float2 *>(leaf_src[pl_.leaf]);
                    default: return out;
                }
            };
            const int32_t accumulate = (nd.is_root && later) ? 1 : 0;
            const uint64_t flops = 8 * nd.m * nd.n * nd.k;
            cudaError_t e;
            if (nd.cls == TN_NODE_DENSE) {
                alignas(128) DenseArgs dargs;
                std::memset(&dargs, 0, sizeof(dargs));
                DenseArgs *d = &dargs;
                const DenseMaps &dm = p->dense_maps[map_of[nd.step]];
                std::memcpy(&d->tmA, &dm.a, sizeof(CUtensorMap));
                std::memcpy(&d->tmB, &dm.b, sizeof(CUtensorMap));
                d->C = resolve(nd.pc);
                // kernel view: rows and columns after the operand swap (the
                // maps were built for that view)
                d->m = (int64_t)dense_rows(nd);
                d->n = (int64_t)dense_cols(nd);
                d->k = (int64_t)nd.k;
                d->lm = nd.swap ? nd.ln : nd.lm;
                d->ln = nd.swap ? nd.lm : nd.ln;
                d->narrow = nd.narrow;
                d->pair = nd.pair;
                d->chunk_kb = (int32_t)(nd.chunk_k /
                                        (p->precision == TN_PREC_BF16 || p->precision == TN_PREC_BF16X3 ? 32 : 16));
                d->accumulate = accumulate;
                d->out_fmt = nd.out_fmt;
                d->out_tile = nd.out_tile;
                d->ktiled = nd.ktiled;
                d->bf16 = p->precision == TN_PREC_BF16;
                d->bf16x3 = p->precision == TN_PREC_BF16X3;
                d->three = nd.three_products;
                d->status = status;
                d->ksplit = nd.ksplit;
                d->kchunk = nd.kchunk;
                d->part = reinterpret_cast<float2 *>(arena + nd.part.off);
                d->ep = nd.ep_off >= 0 ? reinterpret_cast<const EpTable *>(ws + nd.ep_off) : nullptr;
                d->tail_first = nd.tail_first;
                d->tail_cnt = nd.tail_first >= 0 ? reinterpret_cast<int32_t *>(ws + nd.tail_cnt_off)
                                                 : nullptr;
                const uint64_t in_b = fmt_bytes(p->fmt[nd.a]);
                rec.begin(d->bf16x3 ? TN_KERNEL_DENSE_BF16X3
                          : d->bf16 ? TN_KERNEL_DENSE_BF16
                          : d->three ? TN_KERNEL_DENSE_TF32X3_3P : TN_KERNEL_DENSE_TF32X3,
                          nd.step, flops,
                          in_b * (nd.m * nd.k + nd.n * nd.k) +
                              fmt_bytes(nd.out_fmt) * nd.m * nd.n * (accumulate ? 2 : 1));
                e = launch_dense(*d, p->num_sms, dag ? dag->begin() : stream);
                if (dag) dag->end();
                rec.end();
            } else if (nd.cls == TN_NODE_STREAM) {
                StreamArgs a;
                std::memset(&a, 0, sizeof(a));
                // B is the small side: swap operands (C^T = B A^T) when m is
                a.A = resolve(nd.swap ? nd.pb : nd.pa);
                a.B = resolve(nd.swap ? nd.pa : nd.pb);
                a.C = resolve(nd.pc);
                a.part = reinterpret_cast<float2 *>(arena + nd.part.off);
                a.m = (int64_t)(nd.swap ? nd.n : nd.m);
                a.n = (int64_t)(nd.swap ? nd.m : nd.n);
                a.k = (int64_t)nd.k;
                a.kchunk = nd.kchunk;
                a.ksplit = nd.ksplit;
                a.lm = nd.swap ? nd.ln : nd.lm;
                a.ln = nd.swap ? nd.lm : nd.ln;
                a.accumulate = accumulate;
                a.out_fmt = nd.out_fmt;
                a.out_tile = nd.out_tile;
                int lanes;
                int64_t rpc;
                stream_shape((uint64_t)a.m, nd.k, &lanes, &rpc);
                a.lanes = lanes;
                a.rows_per_cta = (int32_t)rpc;
                a.cnt = nd.ksplit > 1 ? reinterpret_cast<int32_t *>(ws + nd.red_cnt_off) : nullptr;
                rec.begin(TN_KERNEL_STREAM, nd.step, flops, node_bytes(nd, accumulate));
                e = launch_stream_node(a, dag ? dag->begin() : stream);
                if (dag) dag->end();
                rec.end();
            } else {
                NodeArgs a;
                std::memset(&a, 0, sizeof(a));
                a.A = resolve(nd.pa);
                a.B = resolve(nd.pb);
                a.C = resolve(nd.pc);
                a.m = (int64_t)nd.m;
                a.n = (int64_t)nd.n;
                a.k = (int64_t)nd.k;
                a.lm = nd.lm;
                a.ln = nd.ln;
                a.accumulate = accumulate;
                a.out_fmt = nd.out_fmt;
                a.out_tile = nd.out_tile;
                a.status = status;
                a.ksplit = nd.ksplit;
                a.kchunk = nd.kchunk;
                a.part = reinterpret_cast<float2 *>(arena + nd.part.off);
                rec.begin(TN_KERNEL_SIMT, nd.step, flops, node_bytes(nd, accumulate));
                e = launch_simt_node(a, dag ? dag->begin() : stream);
                if (dag) dag->end();
                rec.end();
            }
            if (e == cudaSuccess && nd.ksplit > 1 && !fused_reduction(nd)) {
                ReduceArgs r;
                std::memset(&r, 0, sizeof(r));
                const bool sw = nd.swap != 0;   // partials are [split][rows][cols] of the kernel's view
                r.part = reinterpret_cast<const float2 *>(arena + nd.part.off);
                r.C = resolve(nd.pc);
                r.m = (int64_t)(sw ? nd.n : nd.m);
                r.n = (int64_t)(sw ? nd.m : nd.n);
                r.ksplit = nd.ksplit;
                r.lm = sw ? nd.ln : nd.lm;
                r.ln = sw ? nd.lm : nd.ln;
                r.accumulate = accumulate;
                r.out_fmt = nd.out_fmt;
                r.out_tile = nd.out_tile;
                // bytes: every partial read once, the output written once
                rec.begin(TN_KERNEL_REDUCE, nd.step, 0,
                          8 * (uint64_t)nd.ksplit * nd.m * nd.n + fmt_bytes(nd.out_fmt) * nd.m * nd.n);
                e = launch_splitk_reduce(r, dag ? dag->begin() : stream);
                if (dag) dag->end();
                rec.end();
            }
            if (e != cudaSuccess) {
                st = cuda_fail(p, e, "launching a node kernel");
                break;
            }
        }
        if (stop_launch >= 0) break;   // the first slice only
    }
    delete pl;
    return st;
}

}  // namespace

tn_status execute_range(Plan *p, const void *const *leaf_ptrs, void *out_ptr, cudaStream_t stream,
                        uint64_t first, uint64_t step) {
    return issue_range(p, leaf_ptrs, out_ptr, stream, first, step, nullptr);
}

// The first slice's launches up to the one that computes `step`, issued
// directly; its operands and output stay in place for tn_plan_tensor_gather.
tn_status execute_prefix(Plan *p, const void *const *leaf_ptrs, void *out_ptr, int32_t step,
                         cudaStream_t stream) {
    p->prefix_step = -1;
    const int32_t stop = p->launch_of[step];
    if (stop < 0) {
        p->last_error = "step " + std::to_string(step) + " has no launch";
        return TN_EINVAL;
    }
    tn_status st = issue_range(p, leaf_ptrs, out_ptr, stream, 0, 1, nullptr, stop);
    if (st != TN_OK) return st;
    p->prefix_step = step;
    p->prefix_out = out_ptr;
    return TN_OK;
}

// Where tensor `id` of the step tn_execute_prefix stopped at lies, and how.
tn_status tensor_gather(Plan *p, int32_t id, const int64_t *idx, uint64_t count, void *dst,
                        cudaStream_t stream) {
    if (p->prefix_step < 0) {
        p->last_error = "no tn_execute_prefix since the plan was bound or last executed";
        return TN_EINVAL;
    }
    const NodePlan &nd = p->nodes[p->prefix_step];
    if (id != nd.a && id != nd.b && id != nd.out) {
        p->last_error = "tensor " + std::to_string(id) + " is not an operand or the output of step " +
                        std::to_string(p->prefix_step);
        return TN_EINVAL;
    }
    const int n = p->n_tensors;
    // tensors inside a fused group live only in that CTA's shared memory
    // (its leaves are read straight from the caller's buffers): only a
    // group's root reaches memory
    const bool in_group = id < n ? (p->consumer[id] >= 0 && p->fused[p->consumer[id]] >= 0)
                                 : (p->fused[id - n] >= 0 &&
                                    p->fuse_groups[p->fused[id - n]].step != id - n);
    if (in_group) {
        p->last_error = "tensor " + std::to_string(id) +
                        " lives only in the shared memory of a fused leaf subtree";
        return TN_EINVAL;
    }
    GatherArgs g;
    std::memset(&g, 0, sizeof(g));
    Place pl;
    if (id < n) {
        const LeafPlan &lp = p->leaves[id];
        pl = lp.place;
        g.size = lp.size;
        // in place: the caller's complex64 leaf; else the permutation
        // job's destination format and tiling
        g.fmt = FMT_C64;
        g.tile = PlanarTile{0, 0, -1, 0};
        for (size_t j = 0; !lp.in_place && j < p->perm_leaves.size(); ++j)
            if (p->perm_leaves[j] == id) {
                g.tile = p->perm_table[j].tile;
                g.fmt = p->perm_table[j].fmt;
            }
    } else {
        const NodePlan &pr = p->nodes[id - n];
        pl = pr.pc;
        g.size = (int64_t)(pr.m * pr.n);
        g.fmt = pr.out_fmt;
        g.tile = pr.out_tile;
    }
    switch (pl.kind) {
        case PLACE_WS: g.src = static_cast<const char *>(p->ws) + p->arena_off + pl.off; break;
        case PLACE_LEAF: g.src = p->prefix_leaves[pl.leaf]; break;
        default:
            g.src = p->prefix_out;
            g.fmt = FMT_C64;
            g.tile = PlanarTile{0, 0, -1, 0};
    }
    g.idx = idx;
    g.count = (int64_t)count;
    g.dst = static_cast<float2 *>(dst);
    g.status = reinterpret_cast<DevStatus *>(p->ws);
    cudaError_t e = launch_tensor_gather(g, stream);
    return e == cudaSuccess ? TN_OK : cuda_fail(p, e, "launching the tensor gather");
}

// All slices.
tn_status execute_plan(Plan *p, const void *const *leaf_ptrs, void *out_ptr, cudaStream_t stream) {
    return execute_range(p, leaf_ptrs, out_ptr, stream, 0, 1);
}

// tn_execute: the first call with a given (leaves, output, workspace) runs
// the launch sequence directly and then records it, captured on the plan's
// own stream, into a CUDA graph; later calls with the same buffers replay
// the graph on the caller's stream, which removes the host-side launch
// work and most of the gaps between dependent launches.  Profiling runs
// always launch directly.  If capture is unavailable the plan simply keeps
// launching directly.
tn_status execute_replayed(Plan *p, const void *const *leaf_ptrs, void *out_ptr,
                           cudaStream_t stream) {
    if (!p->use_graph || p->profiling) return execute_plan(p, leaf_ptrs, out_ptr, stream);
    // a caller that is capturing its own stream gets the launches recorded
    // into its capture
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
        cudaGetLastError();
        return execute_plan(p, leaf_ptrs, out_ptr, stream);
    }
    const int n = p->n_tensors;
    bool hit = p->graph_exec && p->graph_out == out_ptr && p->graph_ws == p->ws &&
               (int)p->graph_leaves.size() == n;
    for (int t = 0; hit && t < n; ++t) hit = p->graph_leaves[t] == leaf_ptrs[t];
    if (hit) {
        p->prefix_step = -1;
        cudaError_t e = cudaGraphLaunch(static_cast<cudaGraphExec_t>(p->graph_exec), stream);
        if (e != cudaSuccess) return cuda_fail(p, e, "launching the recorded graph");
        return TN_OK;
    }
    drop_graph(p);
    tn_status st = execute_plan(p, leaf_ptrs, out_ptr, stream);
    if (st != TN_OK) return st;
    if (!p->capture_stream) {
        cudaStream_t s;
        if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) {
            cudaGetLastError();
            p->use_graph = false;
            return TN_OK;
        }
        p->capture_stream = s;
    }
    cudaStream_t cs = static_cast<cudaStream_t>(p->capture_stream);
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        cudaGetLastError();
        p->use_graph = false;
        return TN_OK;
    }
    // recorded as a dependency graph: launches that touch no common bytes
    // (independent branches of the tree) may run at the same time
    Dag dag;
    tn_status cst = build_dag(p, cs, 0, 1, &dag);
    if (cst == TN_OK) cst = issue_range(p, leaf_ptrs, out_ptr, cs, 0, 1, &dag);
    if (cst == TN_OK && (dag.next != dag.lane.size() || !dag.join())) cst = TN_ECUDA;
    cudaGraph_t g = nullptr;
    cudaError_t e = cudaStreamEndCapture(cs, &g);
    cudaGraphExec_t ex = nullptr;
    if (cst == TN_OK && e == cudaSuccess && g) e = cudaGraphInstantiate(&ex, g, 0);
    if (g) cudaGraphDestroy(g);
    if (cst != TN_OK || e != cudaSuccess || !ex) {
        cudaGetLastError();
        p->use_graph = false;   // keep launching directly
        return TN_OK;
    }
    p->graph_exec = ex;
    p->graph_leaves.assign(leaf_ptrs, leaf_ptrs + n);
    p->graph_out = out_ptr;
    p->graph_ws = p->ws;
    return TN_OK;
}

// The host call's work on `stream`: leaves in (one gather kernel for
// pinned leaves, a copy for each pageable one), the contraction (replayed,
// or with a recorder its launches), the result out.
tn_status issue_host(Plan *p, const void *const *host_leaves, void *host_out, void *const *dev_leaves,
                     void *dev_out, cudaStream_t stream, Dag *dag) {
    const int n = p->n_tensors;
    GatherLaunch *g = new GatherLaunch;
    g->njobs = 0;
    int ctas = 0;
    cudaError_t e = cudaSuccess;
    auto flush = [&]() {
        if (g->njobs == 0) return;
        g->cta_start[g->njobs] = ctas;
        e = launch_gather(*g, ctas, stream);
        g->njobs = 0;
        ctas = 0;
    };
    for (int t = 0; t < n && e == cudaSuccess; ++t) {
        const int64_t size = p->leaves[t].full_size;
        if (size <= 0) continue;
        if (!p->host_leaves_dev[t]) {
            e = cudaMemcpyAsync(dev_leaves[t], host_leaves[t], (size_t)size * sizeof(float2),
                                cudaMemcpyHostToDevice, stream);
            continue;
        }
        const int j = g->njobs++;
        g->cta_start[j] = ctas;
        g->src[j] = static_cast<const float2 *>(p->host_leaves_dev[t]);
        g->dst[j] = static_cast<float2 *>(dev_leaves[t]);
        g->size[j] = size;
        ctas += permute_ctas(size);
        if (g->njobs == kGatherBatch) flush();
    }
    if (e == cudaSuccess) flush();
    delete g;
    if (e != cudaSuccess) return cuda_fail(p, e, "copying the leaves in");
    const void *const *dl = reinterpret_cast<const void *const *>(dev_leaves);
    tn_status st;
    if (dag) {
        // every lane joins back into `stream` before the result is copied
        st = issue_range(p, dl, dev_out, stream, 0, 1, dag);
        if (st == TN_OK && (dag->next != dag->lane.size() || !dag->join())) st = TN_ECUDA;
    } else {
        st = execute_replayed(p, dl, dev_out, stream);
    }
    if (st != TN_OK) return st;
    e = cudaMemcpyAsync(host_out, dev_out, p->out_elems * sizeof(float2), cudaMemcpyDeviceToHost,
                        stream);
    return e == cudaSuccess ? TN_OK : cuda_fail(p, e, "copying the result out");
}

// tn_execute_host: the caller's host leaves into its device leaf buffers
// (pinned leaves through one gather kernel over their device mappings,
// others by cudaMemcpyAsync), the contraction, the result back to the host.
tn_status execute_host(Plan *p, const void *const *host_leaves, void *host_out,
                       void *const *dev_leaves, void *dev_out, cudaStream_t stream) {
    const int n = p->n_tensors;
    if ((int)p->host_leaves_seen.size() != n) {
        p->host_leaves_seen.assign(n, nullptr);
        p->host_leaves_dev.assign(n, nullptr);
    }
    for (int t = 0; t < n; ++t) {
        if (p->host_leaves_seen[t] == host_leaves[t]) continue;
        cudaPointerAttributes attr;
        const void *dev = nullptr;
        if (cudaPointerGetAttributes(&attr, host_leaves[t]) == cudaSuccess &&
            attr.type == cudaMemoryTypeHost && attr.devicePointer)
            dev = attr.devicePointer;
        cudaGetLastError();   // pageable memory may report an error: not sticky
        p->host_leaves_seen[t] = host_leaves[t];
        p->host_leaves_dev[t] = dev;
    }
    // the whole call as one recorded graph when every buffer on the host
    // side is pinned (copies of pageable memory cannot be recorded)
    bool pinned = true;
    for (int t = 0; t < n; ++t)
        if (p->leaves[t].full_size > 0 && !p->host_leaves_dev[t]) pinned = false;
    if (pinned) {
        cudaPointerAttributes attr;
        pinned = cudaPointerGetAttributes(&attr, host_out) == cudaSuccess && attr.type == cudaMemoryTypeHost;
        cudaGetLastError();
    }
    std::vector<const void *> key(host_leaves, host_leaves + n);
    key.push_back(host_out);
    key.insert(key.end(), dev_leaves, dev_leaves + n);
    key.push_back(dev_out);
    key.push_back(p->ws);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    const bool record = pinned && p->use_graph && !p->profiling &&
                        cudaStreamIsCapturing(stream, &cap) == cudaSuccess && cap == cudaStreamCaptureStatusNone;
    cudaGetLastError();
    p->prefix_step = -1;
    if (record && p->host_graph_exec && p->hg_key == key) {
        cudaError_t e = cudaGraphLaunch(static_cast<cudaGraphExec_t>(p->host_graph_exec), stream);
        return e == cudaSuccess ? TN_OK : cuda_fail(p, e, "launching the recorded host call");
    }
    tn_status st = issue_host(p, host_leaves, host_out, dev_leaves, dev_out, stream, nullptr);
    if (st != TN_OK || !record || !p->use_graph) return st;
    // record the same call on the plan's capture stream for the next time
    if (p->host_graph_exec) cudaGraphExecDestroy(static_cast<cudaGraphExec_t>(p->host_graph_exec));
    p->host_graph_exec = nullptr;
    p->hg_key.clear();
    if (!p->capture_stream) return TN_OK;   // created by the first replayed execute
    cudaStream_t cs = static_cast<cudaStream_t>(p->capture_stream);
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        cudaGetLastError();
        return TN_OK;
    }
    Dag dag;
    tn_status cst = build_dag(p, cs, 0, 1, &dag);
    if (cst == TN_OK) cst = issue_host(p, host_leaves, host_out, dev_leaves, dev_out, cs, &dag);
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(cs, &graph);
    cudaGraphExec_t ex = nullptr;
    if (cst == TN_OK && e == cudaSuccess && graph) e = cudaGraphInstantiate(&ex, graph, 0);
    if (graph) cudaGraphDestroy(graph);
    if (cst != TN_OK || e != cudaSuccess || !ex) {
        cudaGetLastError();   // keep issuing directly
        return TN_OK;
    }
    p->host_graph_exec = ex;
    p->hg_key = key;
    return TN_OK;
}

tn_status read_profile(Plan *p, tn_launch_record *buf, int32_t cap, int32_t *len) {
    const size_t n = p->records.size();
    for (size_t i = 0; i < n; ++i) {
        float ms = 0.f;
        cudaError_t e = cudaEventElapsedTime(&ms, static_cast<cudaEvent_t>(p->events[2 * i]),
                                             static_cast<cudaEvent_t>(p->events[2 * i + 1]));
        if (e != cudaSuccess) return cuda_fail(p, e, "reading launch events");
        p->records[i].ms = ms;
    }
    *len = (int32_t)n;
    for (size_t i = 0; i < n && (int32_t)i < cap; ++i) buf[i] = p->records[i];
    return TN_OK;
}

tn_status check_plan(Plan *p) {
    DevStatus h{0, 0};
    cudaError_t e = cudaMemcpy(&h, p->ws, sizeof(h), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(p, e, "reading the status word");
    if (h.code != ERR_NONE) {
        e = cudaMemset(p->ws, 0, sizeof(h));
        if (e != cudaSuccess) return cuda_fail(p, e, "clearing the status word");
        // a kernel that gave up may have left tail-tile counters raised:
        // restore the tables (counters included) before the next run
        if (!p->table_blob.empty()) {
            e = cudaMemcpy(static_cast<char *>(p->ws) + p->table_off, p->table_blob.data(),
                           p->table_blob.size(), cudaMemcpyHostToDevice);
            if (e != cudaSuccess) return cuda_fail(p, e, "restoring the descriptor tables");
        }
        p->last_error = "device status " + std::to_string(h.code) + " at " + std::to_string(h.where);
        return h.code == ERR_TIMEOUT ? TN_ETIMEOUT : TN_EDEVICE;
    }
    return TN_OK;
}

}  // namespace tn
