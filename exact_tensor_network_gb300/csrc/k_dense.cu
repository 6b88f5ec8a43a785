// Tensor-core node kernel (tcgen05 + TMA + TMEM) for dense pairwise steps.
//
// Computes the step C[i, j] = sum_k A[i, k] * B[j, k] of "Crossing the
// single-GPU memory wall" (section 1.1) in the transpose-free GEMM form
// that lifetime ordering (section 1.4) gives every node: both operands are
// row-major with k fastest ("K-major" in tensor-core terms), so TMA loads
// their tiles as they lie in memory.
//
// Complex arithmetic on real tensor cores.  The producer of each operand
// stores it planar (re and im planes; for the tf32x3 mode each plane is
// also split into hi = tf32(x) and lo = tf32(x - hi), the split-precision
// scheme of Markidis et al. 2018 / Ootomo & Yokota 2022).  A tile of B is
// loaded as the stack [Br; Bi] (256 rows), so one MMA with N = 256 gives
// both Ar*Br and Ar*Bi.  Two TMEM accumulators of 128 lanes x 256 fp32
// columns hold
//     D1 = Ar * [Br; Bi]^T = [ArBr | ArBi],  D2 = Ai * [Br; Bi]^T = [AiBr | AiBi]
// and the epilogue forms Cr = ArBr - AiBi, Ci = ArBi + AiBr.  In tf32x3
// mode each product X*Y is hi*hi + hi*lo + lo*hi (lo*lo dropped).
// Three-product mode (nodes bound by their arithmetic): operands also carry
// the plane s = re + im, and three accumulators of 128 columns hold
//     P1 = Ar Br,  P2 = Ai Bi,  P3 = (Ar + Ai)(Br + Bi)   (N = 128 each)
// so that Cr = P1 - P2 and Ci = P3 - (P1 + P2): 9 instead of 12 tf32 MMAs
// of 128 x 128 per k-step, in exchange for 24-byte operand entries and a
// two-stage ring (96 KiB stages).
//
// Accuracy: the tensor core's fp32 accumulation rounds toward zero, so every
// accumulation into TMEM shrinks the sum a little, always in the same
// direction, and the shrinkage grows with the number of accumulations.  So
// the k range of a tile is cut into chunks (DenseArgs::chunk_kb k-blocks,
// chosen by the planner: 64, 128 or 256 complex k for the split precisions
// depending on how many tensor-core nodes the tree holds, 2048 for plain bf16
// operands); each chunk is accumulated in TMEM from zero, then drained into
// fp32 registers of the epilogue warps with ordinary round-to-nearest adds
// (periodic promotion).  Measured on chains of 2^30-2^32-entry nodes:
// 256-k chunks leave a relative bias of ~1.3e-6 per node, 64-k chunks about
// a quarter of it.
// The two accumulators are handed over separately: the drain reads D1
// while the tensor core runs the last stage's D2 products.
//
// Structure: persistent kernel, one CTA of 384 threads per SM.  Warpgroup
// 0: warp 0 issues TMA loads into a ring of shared-memory stages, warp 1
// issues the MMAs (one thread) and owns the TMEM allocation.  Warpgroups 1
// and 2 (8 warps) drain TMEM: warp w reads TMEM lane quarter w % 4 (rows)
// and one half of the tile's columns, keeps 64 complex running sums per
// thread, and at the end of the tile stores them through the node's
// separable output offsets in the format the consumer wants.  Registers
// are moved from warpgroup 0 to the draining warpgroups with setmaxnreg.
// Output tiles are 128 x 128 complex entries, visited in groups of 8 row
// tiles so that concurrently running CTAs share operand tiles in L2.
// Every wait on an mbarrier is bounded: on timeout the CTA raises an abort
// flag, the roles leave their loops, in-flight copies and MMAs are drained
// (also bounded), TMEM is released and the status word records
// ERR_TIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace tn {

namespace {

constexpr int BM = 128;                 // complex output rows per tile
constexpr int BN = 128;                 // complex output columns per tile
static_assert(BM == kDenseBM && BN == kDenseBN, "tile shape shared with the planner");
constexpr int ROW_BYTES = 64;           // K bytes per smem row (64-byte swizzle)
constexpr int PLANE_TILE = BM * ROW_BYTES;   // 8 KiB: 128 rows of one plane
constexpr int THREADS = 384;            // 3 warpgroups
constexpr int DRAIN_WARPS = 8;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t kTimeoutNs = 4000000000ull;
// register split: launched with 168 per thread (384 x 168 = 64512)
constexpr int REGS_LOW = 56, REGS_HIGH = 224;
static_assert(4 * 32 * REGS_LOW + DRAIN_WARPS * 32 * REGS_HIGH <= THREADS * 168,
              "register split exceeds the launch's registers");

// Kernel modes: split tf32 with four real products per complex product,
// bf16 operands (four products), split tf32 with three products, split
// bf16 (hi and lo bf16 parts, the products hi*hi + hi*lo + lo*hi like the
// split tf32 mode, on the bf16 tensor path).
enum : int { MODE_TF32 = 0, MODE_BF16 = 1, MODE_TF32_3P = 2, MODE_BF16X3 = 3 };

template <int MODE>
struct Cfg {
    static constexpr bool BF16 = MODE == MODE_BF16;
    static constexpr bool THREE = MODE == MODE_TF32_3P;
    static constexpr bool HALF = MODE == MODE_BF16 || MODE == MODE_BF16X3;   // bf16 entries
    // planes per operand: [re, im] (bf16), [re_hi, im_hi, re_lo, im_lo]
    // (tf32 or bf16 parts), or [re_hi, im_hi, s_hi, re_lo, im_lo, s_lo]
    // (s = re + im)
    static constexpr int PLANES = BF16 ? 2 : THREE ? 6 : 4;
    static constexpr int KB = HALF ? 32 : 16;           // complex k per stage
    static constexpr int K_INSTR = HALF ? 16 : 8;       // k per MMA instruction
    // complex k accumulated in TMEM per drain (promotion into fp32 registers)
    static constexpr int CHUNK_K = BF16 ? 256 : 64;
    static constexpr int CHUNK_STAGES = CHUNK_K / KB;
    // CTA pairs accumulate Cr (and Ci) from six products per k-step instead
    // of three per accumulator: half the chunk keeps the same number of
    // accumulations per promotion
    static constexpr int PAIR_CHUNK_K = CHUNK_K / 2;
    static constexpr int PAIR_CHUNK_STAGES = PAIR_CHUNK_K / KB;
    static constexpr int STAGE_BYTES = 2 * PLANES * PLANE_TILE;
    static constexpr int STAGES = BF16 ? 6 : THREE ? 2 : 3;
    // the ring holds 192 KiB in every mode; narrow tiles (B of 64 rows) fit
    // more of their smaller stages into it
    static constexpr int RING = STAGES * STAGE_BYTES;
    static constexpr int NARROW_STAGE_BYTES = PLANES * PLANE_TILE + PLANES * (PLANE_TILE / 2);
    static constexpr int NARROW_STAGES = RING / NARROW_STAGE_BYTES;
    // stages, alignment slack, barriers, then one 32 x 16 complex staging
    // tile per drain warp for coalesced stores
    static constexpr int STAGING = DRAIN_WARPS * 32 * 16 * 8;
    static constexpr int EP_BYTES = (int)((sizeof(EpTable) + 127) / 128 * 128);
    static constexpr int SMEM = RING + 1024 + 256 + STAGING + EP_BYTES;
    // four products: B tiles stacked [Br; Bi] give N = 256 per MMA; three
    // products: each real product is its own N = 128 MMA
    static constexpr uint32_t MMA_N = THREE ? 128 : 256;
    // instruction descriptor without N: D f32, A/B tf32 (2) or bf16 (1),
    // both K-major, M = 128; idesc(N) adds N
    static constexpr uint32_t IDESC_BASE = (1u << 4) | ((HALF ? 1u : 2u) << 7) |
                                           ((HALF ? 1u : 2u) << 10) | ((128u >> 4) << 24);
    static constexpr uint32_t idesc(uint32_t n) { return IDESC_BASE | ((n >> 3) << 17); }
    // CTA pair: M = 256 over the pair, N = 128; bit 13 negates A (the
    // -Ai Bi term of the real part)
    static constexpr uint32_t IDESC_PAIR =
        (IDESC_BASE & ~(0x1Fu << 24)) | ((256u >> 4) << 24) | ((128u >> 3) << 17);
    static constexpr uint32_t IDESC_PAIR_NEG = IDESC_PAIR | (1u << 13);
};
constexpr int MAX_STAGES = 8;   // barrier slots (narrow bf16 tiles: 8 stages)
static_assert(Cfg<MODE_BF16>::NARROW_STAGES <= MAX_STAGES && Cfg<MODE_TF32>::NARROW_STAGES <= MAX_STAGES &&
                  Cfg<MODE_BF16X3>::NARROW_STAGES <= MAX_STAGES,
              "barrier slots");
static_assert(Cfg<MODE_TF32_3P>::SMEM <= 232448 && Cfg<MODE_TF32>::SMEM <= 232448 &&
                  Cfg<MODE_BF16>::SMEM <= 232448 && Cfg<MODE_BF16X3>::SMEM <= 232448,
              "shared memory per CTA");

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with parity `parity`; false if the CTA's abort
// flag is up or the wait ran past the time limit (which raises the flag).
__device__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kTimeoutNs) {
            *abort_flag = 1;
            return false;
        }
    }
}

// Bounded wait that ignores the abort flag (used while draining).
__device__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer() - t0 > kTimeoutNs) return;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// K-tiled operands: one box = one contiguous [128 rows][64 bytes] block.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2, int32_t c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 64-byte swizzle, rows of
// 64 bytes, 8-row core groups 512 bytes apart.
__host__ __device__ constexpr uint64_t sdesc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(512 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(4) << 61);
}
// The same descriptor as two words: the upper one is a constant, the lower
// one holds the address in 16-byte units.  Shared-memory addresses stay
// below 256 KiB, so moving the address by `off` bytes (a multiple of 16)
// adds off / 16 to the lower word without a carry out of its 14-bit field:
// the MMA thread forms a stage's descriptors once and steps them with
// 32-bit adds.
constexpr uint32_t kDescHi = static_cast<uint32_t>(sdesc(0) >> 32);
__host__ __device__ constexpr uint32_t sdesc_lo(uint32_t saddr) {
    return static_cast<uint32_t>(sdesc(saddr));
}
static_assert(sdesc(0x2A3C0) == ((static_cast<uint64_t>(kDescHi) << 32) | sdesc_lo(0x2A3C0)) &&
                  sdesc_lo(0x2A3C0 + 96) == sdesc_lo(0x2A3C0) + 6 &&
                  sdesc_lo(0x37FF0) + 1 == sdesc_lo(0x38000),
              "split descriptor words");

template <int MODE>
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t acc, uint32_t idesc) {
    if constexpr (Cfg<MODE>::HALF) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(acc));
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(acc));
    }
}

// The same MMA from the two descriptor words (lower words of A and B, the
// constant upper word); ACC < 0 takes the accumulate flag from `acc`, else
// it is the constant ACC.
template <int MODE, int ACC>
__device__ __forceinline__ void mma_w(uint32_t d, uint32_t alo, uint32_t blo, uint32_t acc, uint32_t idesc) {
    if constexpr (ACC < 0) {
        if constexpr (Cfg<MODE>::HALF)
            asm volatile(
                "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                "mov.b64 da, {%1, %5};\n\tmov.b64 db, {%2, %5};\n\t"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n\t}" ::"r"(d),
                "r"(alo), "r"(blo), "r"(idesc), "r"(acc), "r"(kDescHi));
        else
            asm volatile(
                "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                "mov.b64 da, {%1, %5};\n\tmov.b64 db, {%2, %5};\n\t"
                "tcgen05.mma.cta_group::1.kind::tf32 [%0], da, db, %3, p;\n\t}" ::"r"(d),
                "r"(alo), "r"(blo), "r"(idesc), "r"(acc), "r"(kDescHi));
    } else {
        if constexpr (Cfg<MODE>::HALF)
            asm volatile(
                "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                "mov.b64 da, {%1, %5};\n\tmov.b64 db, {%2, %5};\n\t"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n\t}" ::"r"(d),
                "r"(alo), "r"(blo), "r"(idesc), "n"(ACC), "r"(kDescHi));
        else
            asm volatile(
                "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                "mov.b64 da, {%1, %5};\n\tmov.b64 db, {%2, %5};\n\t"
                "tcgen05.mma.cta_group::1.kind::tf32 [%0], da, db, %3, p;\n\t}" ::"r"(d),
                "r"(alo), "r"(blo), "r"(idesc), "n"(ACC), "r"(kDescHi));
    }
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// ---- CTA pairs (tcgen05 cta_group::2) ----
// A pair is a cluster of two CTAs on two SMs.  One MMA instruction of the
// leader (rank 0) computes M = 256 rows: rows 0-127 from the leader's shared
// memory and rows 128-255 from the peer's, each CTA holding half of B's N
// rows; each CTA's TMEM receives its own 128 rows.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of both CTAs: shared-memory writes before it are visible to
// the other CTA after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// The same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive on an mbarrier given by its cluster address (possibly the peer's).
// Default (CTA-scope release) semantics: what it orders are the arriving
// warp's TMEM reads, which tcgen05.fence::before_thread_sync already orders
// before it; a cluster-scope release would add a memory barrier per arrive.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

// TMA into this CTA's shared memory, completing on an mbarrier of either
// CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                                 int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                                 int32_t c0, int32_t c1, int32_t c2, int32_t c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

template <int MODE>
__device__ __forceinline__ void mma_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t acc, uint32_t idesc) {
    if constexpr (Cfg<MODE>::HALF) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(acc));
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(acc));
    }
}

// The pair MMA from the two descriptor words (see mma_w).
template <int MODE, int ACC>
__device__ __forceinline__ void mma_pair_w(uint32_t d, uint32_t alo, uint32_t blo, uint32_t acc,
                                           uint32_t idesc) {
    const uint32_t en = ACC < 0 ? acc : static_cast<uint32_t>(ACC);
    if constexpr (Cfg<MODE>::HALF)
        asm volatile(
            "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "mov.b64 da, {%1, %5};\n\tmov.b64 db, {%2, %5};\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %3, p;\n\t}" ::"r"(d),
            "r"(alo), "r"(blo), "r"(idesc), "r"(en), "r"(kDescHi));
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "mov.b64 da, {%1, %5};\n\tmov.b64 db, {%2, %5};\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%0], da, db, %3, p;\n\t}" ::"r"(d),
            "r"(alo), "r"(blo), "r"(idesc), "r"(en), "r"(kDescHi));
}

// Arrive on the mbarrier at this shared-memory offset in both CTAs of the
// pair once the leader's MMAs issued so far have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
    const uint16_t mask = 3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

__device__ __forceinline__ void fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive columns of this thread's TMEM lane (one instruction for
// what two 16-column loads read).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Staging-tile slot of entry e = r * 16 + c of a 32 x 16 block: row r,
// column c xor-swizzled by the row (conflict-light for row and column walks).
__device__ __forceinline__ int swz(int e) { return (e & ~15) | ((e ^ (e >> 4)) & 15); }

// This lane's 16 values of column block cc (a run-time index: the selects
// keep sr / si in registers) into the lane's row of the staging tile.
__device__ __forceinline__ void stage_block(float2 *tile, int lane, const float (&sr)[64],
                                            const float (&si)[64], int cc) {
#pragma unroll
    for (int x = 0; x < 16; ++x) {
        const float vr = cc == 0 ? sr[x] : cc == 1 ? sr[16 + x] : cc == 2 ? sr[32 + x] : sr[48 + x];
        const float vi = cc == 0 ? si[x] : cc == 1 ? si[16 + x] : cc == 2 ? si[32 + x] : si[48 + x];
        tile[swz(lane * 16 + x)] = make_float2(vr, vi);
    }
}

// Work item w of a launch: its tile t, k-block range [kb0, kb1), k split sp
// (split-K) and, for a tail tile's half, which half (else -1).  Work items
// are whole tiles up to tail_first, then two halves per tail tile; with
// split-K, the items of split 0 (every tile), then those of split 1, and so
// on: the CTAs running at the same time then work on the same k range of
// neighbouring tiles and share its operand pieces in L2 (a node with a huge
// k and a few hundred tiles runs many waves; split-by-split, each piece of
// either operand is read from DRAM about once instead of once per wave).
struct Item {
    int64_t t;
    int sp, kb0, kb1, half;
};
__device__ __forceinline__ Item work_item(int64_t w, int ksplit, int kbs, int nkb,
                                          int64_t tail_first, int64_t tiles) {
    Item it;
    it.half = -1;
    if (ksplit > 1) {
        // work < 2^31 items with split-K (tiles x splits is bounded)
        const uint32_t q = static_cast<uint32_t>(w) / static_cast<uint32_t>(tiles);
        it.sp = static_cast<int>(q);
        it.t = static_cast<int64_t>(static_cast<uint32_t>(w) - q * static_cast<uint32_t>(tiles));
        it.kb0 = it.sp * kbs;
        it.kb1 = min(nkb, it.kb0 + kbs);
    } else if (w < tail_first) {
        it.t = w;
        it.sp = 0;
        it.kb0 = 0;
        it.kb1 = nkb;
    } else {
        const int64_t u = w - tail_first;
        it.t = tail_first + (u >> 1);
        it.half = static_cast<int>(u & 1);
        it.sp = 0;
        it.kb0 = it.half ? nkb / 2 : 0;
        it.kb1 = it.half ? nkb : nkb / 2;
    }
    return it;
}

// Output tile of linear tile index t: groups of 8 row tiles, columns inside.
__device__ __forceinline__ void tile_coords(int64_t t, int64_t mtiles, int64_t ntiles, int64_t &mt,
                                            int64_t &nt) {
    const int64_t G = 8;
    const int64_t group = G * ntiles;
    const int64_t g = t / group;
    const int64_t first = g * G;
    const int64_t gm = (mtiles - first) < G ? (mtiles - first) : G;
    const int64_t r = t - g * group;
    mt = first + r % gm;
    nt = r / gm;
}

// Stages in the first promotion chunk of a tile with st k-stages and chunks
// of cs stages.  When a tile starts, the drain is still storing the previous
// tile's outputs; a first chunk of two chunks' length lets the tensor core
// run that long before it needs the drain again, which hides the stores.
// Only tiles of at least eight chunks take it.  A chunk's rounding bias
// grows with its length and weighs by its share of k, so a tile of k = n c
// whose first chunk is 2c has (4 + (n - 2)) / n times the bias of plain
// c-chunks: at most a quarter more (n = 8), an eighth at n = 16.  Measured:
// 4096^3 node +1.4 % (256-k chunks), `circuit_7x7_d10` +2.7 %; the 2^30- and
// 2^32-entry exact-value norm networks' errors 4.0e-6 -> 4.3e-6 and 6.2e-6
// -> 6.4e-6.
__device__ __forceinline__ int first_chunk(int st, int cs) { return st >= 8 * cs ? 2 * cs : cs; }

// The products of one stage into one accumulator of the single-CTA kernel:
// D1 (IM = false) = Ar [Br; Bi] or D2 (IM = true) = Ai [Br; Bi]; split
// precisions form hi*lo + lo*hi + hi*hi.  Fully unrolled with compile-time
// plane offsets: one thread issues every MMA, and its instruction count
// per MMA bounds how fast it can keep the tensor core fed.
template <int MODE, bool IM>
__device__ __forceinline__ void stage_products(uint32_t d, uint32_t base, uint32_t bbase,
                                               uint32_t b_plane, bool fresh, uint32_t idesc) {
    using C = Cfg<MODE>;
    // descriptor lower words of the stage's planes; each instruction takes
    // 32 bytes of K (2 in 16-byte units)
    const uint32_t ah = sdesc_lo(base + (IM ? PLANE_TILE : 0)), bh = sdesc_lo(bbase);
    const uint32_t acc0 = fresh ? 0u : 1u;
    if constexpr (C::BF16) {
        mma_w<MODE, -1>(d, ah, bh, acc0, idesc);
#pragma unroll
        for (int kk = 1; kk < C::KB / C::K_INSTR; ++kk) mma_w<MODE, 1>(d, ah + 2 * kk, bh + 2 * kk, 1, idesc);
    } else {
        const uint32_t al = sdesc_lo(base + (IM ? 3 : 2) * PLANE_TILE), bl = sdesc_lo(bbase + 2 * b_plane);
#pragma unroll
        for (int kk = 0; kk < C::KB / C::K_INSTR; ++kk) {
            if (kk == 0) mma_w<MODE, -1>(d, al, bh, acc0, idesc);
            else mma_w<MODE, 1>(d, al + 2 * kk, bh + 2 * kk, 1, idesc);
            mma_w<MODE, 1>(d, ah + 2 * kk, bl + 2 * kk, 1, idesc);
            mma_w<MODE, 1>(d, ah + 2 * kk, bh + 2 * kk, 1, idesc);
        }
    }
}

// PAIR: the kernel runs as clusters of two CTAs (cta_group::2).  A pair
// owns output tiles of 256 rows x 128 columns: CTA r loads rows
// 128 r .. 128 r + 127 of the tile's A and columns 64 r .. 64 r + 63 of its
// B, the leader issues MMAs of M = 256, N = 128 that form the real and
// imaginary parts directly (Cr = Ar Br - Ai Bi with the negate-A bit,
// Ci = Ar Bi + Ai Br), and each CTA's TMEM holds Cr and Ci of its 128 rows:
// 256 columns, so the accumulators are double-buffered and the drain of one
// chunk overlaps the MMAs of the next.  Each SM reads half as much of B per
// MMA as in the single-CTA kernel.
template <int MODE, bool PAIR>
__global__ void __launch_bounds__(THREADS, 1) dense_kernel(const __grid_constant__ DenseArgs a) {
    using C = Cfg<MODE>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t rank = PAIR ? cluster_rank() : 0;
    // k-blocks accumulated in TMEM per promotion (chosen by the planner)
    const int CS = a.chunk_kb > 0 ? a.chunk_kb : (PAIR ? C::PAIR_CHUNK_STAGES : C::CHUNK_STAGES);
    // narrow tiles (B of 64 rows, smaller stages, more of them, MMA N = 128)
    // and pairs (B of 64 rows per CTA) use the same stage geometry
    const bool narrow = PAIR || (a.narrow && !C::THREE);
    const int stages = narrow ? C::NARROW_STAGES : C::STAGES;
    const int stage_bytes = narrow ? C::NARROW_STAGE_BYTES : C::STAGE_BYTES;
    const int bn = (narrow && !PAIR) ? BN / 2 : BN;   // output columns of a tile
    const int b_plane = narrow ? PLANE_TILE / 2 : PLANE_TILE;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::RING);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + MAX_STAGES);
    // TMEM handoff, per accumulator: full (MMA -> drain), empty (drain -> MMA)
    const uint32_t tmem_full = smem_u32(bars + 2 * MAX_STAGES);
    const uint32_t tmem_empty = smem_u32(bars + 2 * MAX_STAGES + 1);
    const uint32_t drain = smem_u32(bars + 2 * MAX_STAGES + 2);
    const uint32_t tmem_full2 = smem_u32(bars + 2 * MAX_STAGES + 3);
    const uint32_t tmem_empty2 = smem_u32(bars + 2 * MAX_STAGES + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * MAX_STAGES + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        // pairs: the two accumulator buffers; the drain warps of both CTAs
        // release a buffer on the leader's barrier
        mbar_init(tmem_full, 1);
        mbar_init(tmem_empty, PAIR ? 2 * DRAIN_WARPS : DRAIN_WARPS);
        mbar_init(tmem_full2, 1);
        mbar_init(tmem_empty2, PAIR ? 2 * DRAIN_WARPS : DRAIN_WARPS);
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            // one warp of each CTA of the pair allocates together
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_slot)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_slot)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    fence_before();
    __syncthreads();
    // pairs: both CTAs' barriers and TMEM exist before any remote access
    if constexpr (PAIR) cluster_sync();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    // pairs: work items are per pair (the cluster's index)
    const int64_t wfirst = PAIR ? blockIdx.x / 2 : blockIdx.x;
    const int64_t wstride = PAIR ? gridDim.x / 2 : gridDim.x;
    const int64_t tile_rows = PAIR ? 2 * BM : BM;
    // barriers and TMEM are set up (shared memory only); global memory after
    // the previous grid on the stream has completed
    pdl_wait();

    const int64_t mtiles = (a.m + tile_rows - 1) / tile_rows, ntiles = (a.n + bn - 1) / bn;
    const int64_t tiles = mtiles * ntiles;
    const int nkb = static_cast<int>((a.k + C::KB - 1) / C::KB);
    // work item w = (tile w % tiles, k split w / tiles); a split covers kbs
    // k-blocks
    const int ksplit = a.ksplit > 1 ? a.ksplit : 1;
    const int kbs = ksplit > 1 ? static_cast<int>(a.kchunk / C::KB) : nkb;
    // first tail tile and work items: recomputed from the parameters where
    // used, so they hold no registers across the role split
#define TAIL_FIRST ((ksplit == 1 && a.tail_first >= 0) ? a.tail_first : tiles)
#define WORK (ksplit > 1 ? tiles * ksplit : TAIL_FIRST + 2 * (tiles - TAIL_FIRST))

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_LOW));
        if (warp == 0 && lane == 0) {
            // ---- TMA producer ----
            uint32_t stage = 0, phase = 0;
            uint32_t issued = 0, last_par = 0;   // bit s: stage s has a load; its parity
            bool ok = true;
            for (int64_t w = wfirst; w < WORK && ok; w += wstride) {
                const Item it = work_item(w, ksplit, kbs, nkb, TAIL_FIRST, tiles);
                int64_t mt, nt;
                tile_coords(it.t, mtiles, ntiles, mt, nt);
                // pairs: this CTA's 128 rows of A and 64 rows (columns of the
                // tile) of B
                const int32_t ym = static_cast<int32_t>(mt * tile_rows + rank * BM);
                const int32_t yn = static_cast<int32_t>(nt * bn + (PAIR ? rank * (BN / 2) : 0));
                const int kb0 = it.kb0, kb1 = it.kb1;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bounded(empty0 + 8 * stage, phase ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint32_t bar = full0 + 8 * stage;
                    if constexpr (PAIR) {
                        // the leader's barrier counts both CTAs' bytes
                        if (rank == 0) mbar_expect_tx(bar, 2 * stage_bytes);
                        bar = map_to_rank(bar, 0);
                    } else {
                        mbar_expect_tx(bar, stage_bytes);
                    }
                    const uint32_t base = smem_u32(smem + stage * stage_bytes);
                    const int32_t kx = kb * C::KB;
                    // B planes in the same order land as the stacks [re; im]
                    // of each split part (hi stack, then lo stack)
                    const uint32_t bbase = base + C::PLANES * PLANE_TILE;
                    if (a.ktiled) {
#pragma unroll
                        for (int p = 0; p < C::PLANES; ++p) {
                            if constexpr (PAIR) {
                                tma_load_4d_pair(base + p * PLANE_TILE, &a.tmA, bar, 0, ym, kb, p);
                                tma_load_4d_pair(bbase + p * b_plane, &a.tmB, bar, 0, yn, kb, p);
                            } else {
                                tma_load_4d(base + p * PLANE_TILE, &a.tmA, bar, 0, ym, kb, p);
                                tma_load_4d(bbase + p * b_plane, &a.tmB, bar, 0, yn, kb, p);
                            }
                        }
                    } else {
#pragma unroll
                        for (int p = 0; p < C::PLANES; ++p) {
                            if constexpr (PAIR) {
                                tma_load_3d_pair(base + p * PLANE_TILE, &a.tmA, bar, kx, ym, p);
                                tma_load_3d_pair(bbase + p * b_plane, &a.tmB, bar, kx, yn, p);
                            } else {
                                tma_load_3d(base + p * PLANE_TILE, &a.tmA, bar, kx, ym, p);
                                tma_load_3d(bbase + p * b_plane, &a.tmB, bar, kx, yn, p);
                            }
                        }
                    }
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // copies in flight complete before the CTA leaves (pairs: the
            // leader's barriers count the peer's copies too)
            if (!ok && rank == 0) {
                for (int s = 0; s < stages; ++s)
                    if (issued & (1u << s)) drain_wait(full0 + 8 * s, (last_par >> s) & 1);
            }
        } else if (PAIR && warp == 1 && lane == 0 && rank == 0) {
            // ---- MMA issuer of a pair ----
            // buffer b (chunks alternate): Cr at column 256 b, Ci at 256 b + 128
            uint32_t stage = 0, phase = 0, cnt = 0;
            bool ok = true;
            for (int64_t w = wfirst; w < WORK && ok; w += wstride) {
                const Item it = work_item(w, ksplit, kbs, nkb, TAIL_FIRST, tiles);
                const int kb0 = it.kb0, kb1 = it.kb1;
                const int nch = (kb1 - kb0 + CS - 1) / CS;
                for (int ch = 0; ch < nch && ok; ++ch, ++cnt) {
                    const uint32_t b = cnt & 1, ph = (cnt >> 1) & 1;
                    // both CTAs' drains have read this buffer's last chunk
                    if (!wait_bounded(b ? tmem_empty2 : tmem_empty, ph ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t cr = tmem + 256 * b, ci = cr + 128;
                    const int kb_beg = kb0 + ch * CS;
                    const int kb_end = min(kb1, kb_beg + CS);
                    for (int kb = kb_beg; kb < kb_end; ++kb) {
                        if (!wait_bounded(full0 + 8 * stage, phase, abort_flag)) {
                            ok = false;
                            break;
                        }
                        fence_after();
                        const uint32_t base = smem_u32(smem + stage * stage_bytes);
                        const uint32_t bbase = base + C::PLANES * PLANE_TILE;
                        const uint32_t acc0 = kb == kb_beg ? 0u : 1u;
                        constexpr uint32_t id = C::IDESC_PAIR, idn = C::IDESC_PAIR_NEG;
                        // descriptor lower words of the stage's planes, stepped
                        // by 2 (32 bytes of K) per instruction
                        const uint32_t arh = sdesc_lo(base), aih = sdesc_lo(base + PLANE_TILE);
                        const uint32_t brh = sdesc_lo(bbase), bih = sdesc_lo(bbase + b_plane);
                        if constexpr (C::BF16) {
#pragma unroll
                            for (int kk = 0; kk < C::KB / C::K_INSTR; ++kk) {
                                const uint32_t o = 2 * kk;
                                if (kk == 0) {
                                    mma_pair_w<MODE, -1>(cr, arh, brh, acc0, id);
                                    mma_pair_w<MODE, 1>(cr, aih, bih, 1, idn);   // - Ai Bi
                                    mma_pair_w<MODE, -1>(ci, arh, bih, acc0, id);
                                } else {
                                    mma_pair_w<MODE, 1>(cr, arh + o, brh + o, 1, id);
                                    mma_pair_w<MODE, 1>(cr, aih + o, bih + o, 1, idn);
                                    mma_pair_w<MODE, 1>(ci, arh + o, bih + o, 1, id);
                                }
                                mma_pair_w<MODE, 1>(ci, aih + o, brh + o, 1, id);
                            }
                        } else {
                            // planes [re_hi, im_hi, re_lo, im_lo]; each product
                            // is hi*lo + lo*hi + hi*hi
                            const uint32_t arl = sdesc_lo(base + 2 * PLANE_TILE), ail = sdesc_lo(base + 3 * PLANE_TILE);
                            const uint32_t brl = sdesc_lo(bbase + 2 * b_plane), bil = sdesc_lo(bbase + 3 * b_plane);
#pragma unroll
                            for (int kk = 0; kk < C::KB / C::K_INSTR; ++kk) {
                                const uint32_t o = 2 * kk;
                                if (kk == 0) {
                                    mma_pair_w<MODE, -1>(cr, arl, brh, acc0, id);
                                } else {
                                    mma_pair_w<MODE, 1>(cr, arl + o, brh + o, 1, id);
                                }
                                mma_pair_w<MODE, 1>(cr, arh + o, brl + o, 1, id);
                                mma_pair_w<MODE, 1>(cr, arh + o, brh + o, 1, id);
                                mma_pair_w<MODE, 1>(cr, ail + o, bih + o, 1, idn);
                                mma_pair_w<MODE, 1>(cr, aih + o, bil + o, 1, idn);
                                mma_pair_w<MODE, 1>(cr, aih + o, bih + o, 1, idn);
                                if (kk == 0) {
                                    mma_pair_w<MODE, -1>(ci, arl, bih, acc0, id);
                                } else {
                                    mma_pair_w<MODE, 1>(ci, arl + o, bih + o, 1, id);
                                }
                                mma_pair_w<MODE, 1>(ci, arh + o, bil + o, 1, id);
                                mma_pair_w<MODE, 1>(ci, arh + o, bih + o, 1, id);
                                mma_pair_w<MODE, 1>(ci, ail + o, brh + o, 1, id);
                                mma_pair_w<MODE, 1>(ci, aih + o, brl + o, 1, id);
                                mma_pair_w<MODE, 1>(ci, aih + o, brh + o, 1, id);
                            }
                        }
                        mma_commit_pair(empty0 + 8 * stage);   // both CTAs may refill the stage
                        if (++stage == stages) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                    if (!ok) break;
                    mma_commit_pair(b ? tmem_full2 : tmem_full);   // both drains may read
                }
            }
            mma_commit_pair(drain);
            drain_wait(drain, 0);
        } else if (!PAIR && !C::THREE && warp == 1 && lane == 0) {
            // ---- MMA issuer (single CTA) ----
            // D1 = Ar [Br; Bi] and D2 = Ai [Br; Bi], 2 bn columns each, are
            // promoted in chunks of CS stages, ending at the same stages; each
            // is committed to the drain right after its own products, so the
            // drain reads D1 while the tensor core runs the stage's D2
            // products.  (Boundaries of D2 offset from D1's, so that each
            // accumulator's drain hides behind two stages of the other's
            // products, measured 1-3 % slower on 4096^3 nodes and up to a
            // third slower on tiles of one or two chunks.)
            const uint32_t d1 = tmem, d2 = tmem + 2 * bn;
            const uint32_t idesc = C::idesc((uint32_t)(2 * bn));
            uint32_t stage = 0, phase = 0, ph1 = 0, ph2 = 0;
            bool ok = true;
            for (int64_t w = wfirst; w < WORK && ok; w += wstride) {
                const Item it = work_item(w, ksplit, kbs, nkb, TAIL_FIRST, tiles);
                const int kb0 = it.kb0, kb1 = it.kb1;
                // stage within the chunk, stepped without a division; the
                // first chunk of a long tile is two chunks (first_chunk)
                int cpos = 0, clen = first_chunk(kb1 - kb0, CS);
                for (int kb = kb0; kb < kb1 && ok; ++kb) {
                    const bool cstart = cpos == 0, cend = cpos == clen - 1 || kb == kb1 - 1;
                    if (cpos == clen - 1) {
                        cpos = 0;
                        clen = CS;
                    } else {
                        ++cpos;
                    }
                    if (!wait_bounded(full0 + 8 * stage, phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t base = smem_u32(smem + stage * stage_bytes);
                    const uint32_t bbase = base + C::PLANES * PLANE_TILE;
                    if (cstart) {
                        if (!wait_bounded(tmem_empty, ph1 ^ 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        fence_after();
                    }
                    stage_products<MODE, false>(d1, base, bbase, b_plane, cstart, idesc);
                    if (cend) {
                        mma_commit(tmem_full);    // the drain may read D1
                        ph1 ^= 1;
                    }
                    if (cstart) {
                        if (!wait_bounded(tmem_empty2, ph2 ^ 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        fence_after();
                    }
                    stage_products<MODE, true>(d2, base, bbase, b_plane, cstart, idesc);
                    if (cend) {
                        mma_commit(tmem_full2);   // the drain may read D2
                        ph2 ^= 1;
                    }
                    if (!ok) break;
                    mma_commit(empty0 + 8 * stage);
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            mma_commit(drain);
            drain_wait(drain, 0);
        } else if (!PAIR && C::THREE && warp == 1 && lane == 0) {
            // ---- MMA issuer ----
            // four products: D1 = Ar [Br; Bi], D2 = Ai [Br; Bi], 2 bn columns each
            const uint32_t d1 = tmem, d2 = tmem + 2 * bn;
            const uint32_t idesc = C::idesc(C::THREE ? 128u : (uint32_t)(2 * bn));
            uint32_t stage = 0, phase = 0, tphase = 0;
            bool ok = true;
            for (int64_t w = wfirst; w < WORK && ok; w += wstride) {
                const Item it = work_item(w, ksplit, kbs, nkb, TAIL_FIRST, tiles);
                const int kb0 = it.kb0, kb1 = it.kb1;
                const int nch = (kb1 - kb0 + CS - 1) / CS;
                for (int ch = 0; ch < nch && ok; ++ch) {
                    // D1 must have been read by the drain (three products:
                    // every accumulator, both halves)
                    if (!wait_bounded(tmem_empty, tphase ^ 1, abort_flag) ||
                        (C::THREE && !wait_bounded(tmem_empty2, tphase ^ 1, abort_flag))) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    bool d2_free = C::THREE;
                    const int kb_beg = kb0 + ch * CS;
                    const int kb_end = min(kb1, kb_beg + CS);
                    for (int kb = kb_beg; kb < kb_end; ++kb) {
                        if (!wait_bounded(full0 + 8 * stage, phase, abort_flag)) {
                            ok = false;
                            break;
                        }
                        fence_after();
                        const uint32_t base = smem_u32(smem + stage * stage_bytes);
                        const uint32_t bbase = base + C::PLANES * PLANE_TILE;
                        const bool first = kb == kb_beg;
                        const bool last = kb == kb_end - 1;
                        // D1: the products of A's real planes (three products:
                        // all of them)
#pragma unroll
                        for (int kk = 0; kk < C::KB / C::K_INSTR; ++kk) {
                            const uint32_t off = kk * 32;   // 32 bytes of K per instruction
                            const uint32_t acc = (first && kk == 0) ? 0u : 1u;
                            if constexpr (C::BF16) {
                                mma<MODE>(d1, sdesc(base + off), sdesc(bbase + off), acc, idesc);
                            } else if constexpr (C::THREE) {
                                // D_c (128 columns at 128 c) = A_c B_c for the
                                // components c = re, im, re + im
#pragma unroll
                                for (int c = 0; c < 3; ++c) {
                                    const uint32_t dc = tmem + 128 * c;
                                    const uint64_t ah = sdesc(base + c * PLANE_TILE + off);
                                    const uint64_t al = sdesc(base + (c + 3) * PLANE_TILE + off);
                                    const uint64_t bh = sdesc(bbase + c * PLANE_TILE + off);
                                    const uint64_t bl = sdesc(bbase + (c + 3) * PLANE_TILE + off);
                                    mma<MODE>(dc, al, bh, acc, idesc);
                                    mma<MODE>(dc, ah, bl, 1, idesc);
                                    mma<MODE>(dc, ah, bh, 1, idesc);
                                }
                            } else {
                                const uint64_t arh = sdesc(base + off);
                                const uint64_t arl = sdesc(base + 2 * PLANE_TILE + off);
                                const uint64_t bh = sdesc(bbase + off);
                                const uint64_t bl = sdesc(bbase + 2 * b_plane + off);
                                mma<MODE>(d1, arl, bh, acc, idesc);
                                mma<MODE>(d1, arh, bl, 1, idesc);
                                mma<MODE>(d1, arh, bh, 1, idesc);
                            }
                        }
                        if (last) mma_commit(tmem_full);   // the drain may read D1
                        if (!d2_free) {
                            // the drain releases D2 while these D1 products run
                            if (!wait_bounded(tmem_empty2, tphase ^ 1, abort_flag)) {
                                ok = false;
                                break;
                            }
                            fence_after();
                            d2_free = true;
                        }
                        // D2: the products of A's imaginary planes
                        if constexpr (!C::THREE) {
#pragma unroll
                            for (int kk = 0; kk < C::KB / C::K_INSTR; ++kk) {
                                const uint32_t off = kk * 32;
                                const uint32_t acc = (first && kk == 0) ? 0u : 1u;
                                if constexpr (C::BF16) {
                                    mma<MODE>(d2, sdesc(base + PLANE_TILE + off), sdesc(bbase + off),
                                              acc, idesc);
                                } else {
                                    const uint64_t aih = sdesc(base + PLANE_TILE + off);
                                    const uint64_t ail = sdesc(base + 3 * PLANE_TILE + off);
                                    const uint64_t bh = sdesc(bbase + off);
                                    const uint64_t bl = sdesc(bbase + 2 * b_plane + off);
                                    mma<MODE>(d2, ail, bh, acc, idesc);
                                    mma<MODE>(d2, aih, bl, 1, idesc);
                                    mma<MODE>(d2, aih, bh, 1, idesc);
                                }
                            }
                        }
                        mma_commit(empty0 + 8 * stage);
                        if (last) mma_commit(tmem_full2);   // the drain may read D2
                        if (++stage == stages) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                    if (!ok) break;
                    tphase ^= 1;
                }
            }
            mma_commit(drain);
            drain_wait(drain, 0);
        }
        __syncwarp();
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_HIGH));
        // ---- drain: TMEM chunks -> fp32 running sums -> global ----
        const int q = warp & 3;                 // TMEM lane quarter (rows)
        const int h = (warp - 4) >> 2;          // column half of the tile
        const int half_cols = bn / 2;           // columns per drain warp (64, narrow 32)
        const int ncc = bn / 32;                // 16-column blocks per drain warp
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const int64_t plane = a.m * a.n;
        const int nl = a.ln.nrun;
        const int64_t last_ext = nl > 0 ? a.ln.ext[nl - 1] : 1;
        const int64_t last_stride = nl > 0 ? a.ln.stride[nl - 1] : 0;
        // split-K partials are plain row-major C64; otherwise the node's
        // output.  When consecutive rows are adjacent in the output (its
        // fastest mode is in M) thread-per-row stores coalesce as they are;
        // otherwise each warp transposes 32 x 16 blocks through shared memory
        // so that 16 lanes store 16 consecutive columns.
        const bool plain = ksplit > 1;
        const bool rows_adjacent =
            !plain && a.lm.nrun > 0 && a.lm.stride[a.lm.nrun - 1] == 1;
        const int32_t fmt = plain ? (int32_t)FMT_C64 : a.out_fmt;
        const int32_t accum = plain ? 0 : a.accumulate;
        float2 *stage_tile = reinterpret_cast<float2 *>(
            smem + C::RING + 256 + (warp - 4) * 32 * 16 * 8);
        EpTable *ep_s = nullptr;
        if (a.ep && !plain) {
            ep_s = reinterpret_cast<EpTable *>(smem + C::RING + 256 + C::STAGING);
            const uint32_t *src = reinterpret_cast<const uint32_t *>(a.ep);
            uint32_t *dstw = reinterpret_cast<uint32_t *>(ep_s);
            for (int x = threadIdx.x - 128; x < (int)(sizeof(EpTable) / 4); x += DRAIN_WARPS * 32)
                dstw[x] = src[x];
            asm volatile("bar.sync 1, %0;" ::"n"(DRAIN_WARPS * 32) : "memory");
        }
        // pretiled tables hold tiled offsets: tile the block base only
        const bool pretiled = ep_s && ep_s->pretiled;
        // runs of four need a 16-byte aligned destination (the caller's
        // output may not be)
        const bool quads =
            ep_s && ep_s->vec && (reinterpret_cast<uintptr_t>(a.C) & 15) == 0;
        const PlanarTile ep_tile = pretiled ? PlanarTile{0, 0, -1, 0} : a.out_tile;
        uint32_t tphase = 0, pcnt = 0, q1 = 0, q2 = 0;
        bool ok = true;
        for (int64_t w = wfirst; w < WORK && ok; w += wstride) {
            const Item it = work_item(w, ksplit, kbs, nkb, TAIL_FIRST, tiles);
            const int sp = it.sp;
            const int kb0 = it.kb0, kb1 = it.kb1;
            const int nch = (kb1 - kb0 + CS - 1) / CS;
            int64_t mt, nt;
            tile_coords(it.t, mtiles, ntiles, mt, nt);
            float sr[64], si[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) sr[c] = si[c] = 0.f;
            if constexpr (PAIR) {
                // buffer b of chunk cnt holds Cr and Ci of this CTA's rows
                for (int ch = 0; ch < nch; ++ch, ++pcnt) {
                    const uint32_t b = pcnt & 1, ph = (pcnt >> 1) & 1;
                    int okv = 0;
                    if (lane == 0) okv = wait_bounded(b ? tmem_full2 : tmem_full, ph, abort_flag) ? 1 : 0;
                    okv = __shfl_sync(0xffffffffu, okv, 0);
                    if (!okv) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t cr = lane_base + 256 * b, ci = cr + 128;
#pragma unroll
                    for (int cp = 0; cp < 4; cp += 2) {
                        const uint32_t col = h * half_cols + cp * 16;
                        float r0[16], i0v[16], r1[16], i1v[16];
                        tmem_ld16(cr + col, r0);
                        tmem_ld16(ci + col, i0v);
                        tmem_ld16(cr + col + 16, r1);
                        tmem_ld16(ci + col + 16, i1v);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            sr[cp * 16 + c] += r0[c];
                            si[cp * 16 + c] += i0v[c];
                            sr[cp * 16 + 16 + c] += r1[c];
                            si[cp * 16 + 16 + c] += i1v[c];
                        }
                    }
                    fence_before();
                    __syncwarp();
                    // release the buffer on the leader's barrier
                    if (lane == 0) mbar_arrive_cluster(map_to_rank(b ? tmem_empty2 : tmem_empty, 0));
                }
            }
            if constexpr (!PAIR && !C::THREE) {
                // the chunks of D1 and D2 alternate, D1 first (see the MMA
                // issuer)
                const int st = kb1 - kb0, f = first_chunk(st, CS);
                const int nch2 = 2 * (st <= f ? 1 : 1 + (st - f + CS - 1) / CS);
                for (int e = 0; e < nch2; ++e) {
                    const bool im = (e & 1) == 1;
                    int okv = 0;
                    if (lane == 0)
                        okv = wait_bounded(im ? tmem_full2 : tmem_full, im ? q2 : q1, abort_flag) ? 1 : 0;
                    okv = __shfl_sync(0xffffffffu, okv, 0);
                    if (!okv) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    // D1 = [ArBr | ArBi]: re += ArBr, im += ArBi; D2 = [AiBr | AiBi]:
                    // re -= AiBi, im += AiBr.  Two column blocks (two 32-column
                    // loads) in flight per round
                    const uint32_t dcol = im ? 2 * bn : 0;
#pragma unroll
                    for (int cp = 0; cp < 4; cp += 2) {
                        if (cp >= ncc) break;   // warp-uniform (narrow tiles: 2 blocks)
                        const uint32_t col = dcol + h * half_cols + cp * 16;
                        float xr[32], xi[32];
                        tmem_ld32(lane_base + col, xr);
                        tmem_ld32(lane_base + bn + col, xi);
                        tmem_wait_ld();
                        if (im) {
#pragma unroll
                            for (int c = 0; c < 32; ++c) {
                                sr[cp * 16 + c] -= xi[c];
                                si[cp * 16 + c] += xr[c];
                            }
                        } else {
#pragma unroll
                            for (int c = 0; c < 32; ++c) {
                                sr[cp * 16 + c] += xr[c];
                                si[cp * 16 + c] += xi[c];
                            }
                        }
                    }
                    fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(im ? tmem_empty2 : tmem_empty);
                    if (im) q2 ^= 1;
                    else q1 ^= 1;
                }
            }
            for (int ch = 0; !PAIR && C::THREE && ch < nch; ++ch) {
                int okv = 0;
                if (lane == 0) okv = wait_bounded(tmem_full, tphase, abort_flag) ? 1 : 0;
                okv = __shfl_sync(0xffffffffu, okv, 0);
                if (!okv) {
                    ok = false;
                    break;
                }
                fence_after();
                if constexpr (C::THREE) {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        if (cc >= ncc) break;   // warp-uniform
                        const uint32_t col = h * half_cols + cc * 16;
                        // P1 = ArBr, P2 = AiBi, P3 = (Ar + Ai)(Br + Bi):
                        // re = P1 - P2, im = P3 - (P1 + P2)
                        float p1[16], p2[16], p3[16];
                        tmem_ld16(lane_base + col, p1);
                        tmem_ld16(lane_base + 128 + col, p2);
                        tmem_ld16(lane_base + 256 + col, p3);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            sr[cc * 16 + c] += p1[c] - p2[c];
                            si[cc * 16 + c] += p3[c] - (p1[c] + p2[c]);
                        }
                    }
                } else {
                    // D1 = [ArBr | ArBi]: two column blocks (four loads) in
                    // flight per round
#pragma unroll
                    for (int cp = 0; cp < 4; cp += 2) {
                        if (cp >= ncc) break;   // warp-uniform (narrow tiles: 2 blocks)
                        const uint32_t col = h * half_cols + cp * 16;
                        float rr0[16], ri0[16], rr1[16], ri1[16];
                        tmem_ld16(lane_base + col, rr0);
                        tmem_ld16(lane_base + bn + col, ri0);
                        tmem_ld16(lane_base + col + 16, rr1);
                        tmem_ld16(lane_base + bn + col + 16, ri1);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            sr[cp * 16 + c] += rr0[c];
                            si[cp * 16 + c] += ri0[c];
                            sr[cp * 16 + 16 + c] += rr1[c];
                            si[cp * 16 + 16 + c] += ri1[c];
                        }
                    }
                }
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tmem_empty);   // D1 may be overwritten
                if (lane == 0) okv = wait_bounded(tmem_full2, tphase, abort_flag) ? 1 : 0;
                okv = __shfl_sync(0xffffffffu, okv, 0);
                if (!okv) {
                    ok = false;
                    break;
                }
                fence_after();
                if constexpr (!C::THREE) {
                    // D2 = [AiBr | AiBi]: re -= AiBi, im += AiBr
#pragma unroll
                    for (int cp = 0; cp < 4; cp += 2) {
                        if (cp >= ncc) break;
                        const uint32_t col = h * half_cols + cp * 16;
                        float ir0[16], ii0[16], ir1[16], ii1[16];
                        tmem_ld16(lane_base + 2 * bn + col, ir0);
                        tmem_ld16(lane_base + 3 * bn + col, ii0);
                        tmem_ld16(lane_base + 2 * bn + col + 16, ir1);
                        tmem_ld16(lane_base + 3 * bn + col + 16, ii1);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            sr[cp * 16 + c] -= ii0[c];
                            si[cp * 16 + c] += ir0[c];
                            sr[cp * 16 + 16 + c] -= ii1[c];
                            si[cp * 16 + 16 + c] += ir1[c];
                        }
                    }
                }
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tmem_empty2);   // D2 may be overwritten
                tphase ^= 1;
            }
            if (!ok) break;
            // A tail tile's half.  Each drain warp pairs with the same warp
            // (same 32 x 64 block) of the other half's CTA: it publishes its
            // sums and counts in; the second to arrive adds the other's sums
            // (below, block by block) and stores.  Two terms: the sum is the
            // same whichever comes first.  Per warp: no wait on another warp
            // or CTA.
            const float2 *other = nullptr;
            if (it.half >= 0) {
                const int64_t slot = (it.t - TAIL_FIRST) * DRAIN_WARPS + (warp - 4);
                float2 *mine = a.part + (slot * 2 + it.half) * (64 * 32);
                // through the staging tile, block by block (rolled: unrolled
                // stores of all 64 sums would spill registers)
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    stage_block(stage_tile, lane, sr, si, cc);
#pragma unroll 4
                    for (int x = 0; x < 16; ++x)
                        mine[(cc * 16 + x) * 32 + lane] = stage_tile[swz(lane * 16 + x)];
                    __syncwarp();
                }
                __threadfence();
                __syncwarp();
                int first = 0;
                if (lane == 0) first = atomicAdd(a.tail_cnt + slot, 1) == 0;
                first = __shfl_sync(0xffffffffu, first, 0);
                if (first) continue;
                __threadfence();
                if (lane == 0) a.tail_cnt[slot] = 0;   // ready for the next run
                other = a.part + (slot * 2 + (it.half ^ 1)) * (64 * 32);
            }
            void *dst = plain ? static_cast<void *>(a.part + (int64_t)sp * plane) : a.C;
            const int64_t i0 = mt * tile_rows + rank * BM + q * 32;
            const int64_t i = i0 + lane;
            const int64_t offm = i < a.m ? (plain ? i * a.n : sep_offset(a.lm, i)) : 0;
            const int64_t bm = ep_s ? sep_offset(a.lm, i0) : 0;
            // One 32 x 16 block (this warp's rows, 16 columns) per pass.  The
            // block goes through the staging tile (row = lane, columns
            // xor-swizzled by row) and every store loop reads it from there,
            // so the loops stay rolled and the kernel's code stays small.
#pragma unroll 1
            for (int cc = 0; cc < ncc; ++cc) {
                const int64_t j0 = nt * bn + h * half_cols + cc * 16;
                if (j0 >= a.n) break;   // warp-uniform
                stage_block(stage_tile, lane, sr, si, cc);
                if (other) {
                    // the other half's sums of this lane's 16 entries
#pragma unroll 4
                    for (int x = 0; x < 16; ++x) {
                        const float2 v = __ldcg(other + (cc * 16 + x) * 32 + lane);
                        float2 &d = stage_tile[swz(lane * 16 + x)];
                        d.x += v.x;
                        d.y += v.y;
                    }
                }
                __syncwarp();
                if (ep_s) {
                    // the block in address order
                    int64_t base = bm + sep_offset(a.ln, j0);
                    if (pretiled) base = tiled_offset(a.out_tile, base);
                    if (quads && i0 + 32 <= a.m && j0 + 16 <= a.n) {   // warp-uniform
                        // each lane stores a run of four consecutive entries
                        const uint2 *pk = reinterpret_cast<const uint2 *>(ep_s->perm);
#pragma unroll 1
                        for (int it = 0; it < 4; ++it) {
                            const uint2 w4 = pk[it * 32 + lane];
                            const int e0 = (int)(w4.x & 0xffffu), e1 = (int)(w4.x >> 16);
                            const int e2 = (int)(w4.y & 0xffffu), e3 = (int)(w4.y >> 16);
                            const float2 v[4] = {stage_tile[swz(e0)], stage_tile[swz(e1)],
                                                 stage_tile[swz(e2)], stage_tile[swz(e3)]};
                            store_quad(dst, fmt, plane,
                                       base + ep_s->lo_m[e0 >> 4] + ep_s->lo_n[e0 & 15], v, accum,
                                       ep_tile);
                        }
                    } else {
#pragma unroll 1
                        for (int it = 0; it < 16; ++it) {
                            const int e = ep_s->perm[it * 32 + lane];
                            const int r = e >> 4, c = e & 15;
                            if (i0 + r < a.m && j0 + c < a.n)
                                store_entry(dst, fmt, plane, base + ep_s->lo_m[r] + ep_s->lo_n[c],
                                            stage_tile[swz(e)], accum, ep_tile);
                        }
                    }
                } else if (rows_adjacent) {
                    // thread per row: consecutive lanes are consecutive entries
                    if (i < a.m) {
                        const bool fast = (j0 % last_ext) + 16 <= last_ext;
                        const int64_t offn0 = sep_offset(a.ln, j0);
#pragma unroll 1
                        for (int c = 0; c < 16 && j0 + c < a.n; ++c) {
                            const int64_t offn =
                                fast ? offn0 + c * last_stride : sep_offset(a.ln, j0 + c);
                            store_entry(dst, fmt, plane, offm + offn, stage_tile[swz(lane * 16 + c)],
                                        accum, a.out_tile);
                        }
                    }
                } else {
                    // 16 lanes store 16 consecutive columns of two rows
                    const int c = lane & 15;
                    const int64_t j = j0 + c;
                    int64_t offn = 0;
                    if (j < a.n) {
                        if (plain) {
                            offn = j;
                        } else {
                            const bool fast = (j0 % last_ext) + 16 <= last_ext;
                            offn = fast ? sep_offset(a.ln, j0) + c * last_stride : sep_offset(a.ln, j);
                        }
                    }
#pragma unroll 1
                    for (int it = 0; it < 16; ++it) {
                        const int r = 2 * it + (lane >> 4);
                        const int64_t om = __shfl_sync(0xffffffffu, offm, r);
                        if (i0 + r < a.m && j < a.n)
                            store_entry(dst, fmt, plane, om + offn, stage_tile[swz(r * 16 + c)], accum,
                                        a.out_tile);
                    }
                }
                __syncwarp();
            }
        }
    }

#undef WORK
#undef TAIL_FIRST
    fence_before();
    __syncthreads();
    // pairs: neither CTA leaves (or frees TMEM) while the other may still
    // reach its shared memory or TMEM
    if constexpr (PAIR) cluster_sync();
    if (warp == 1) {
        fence_after();
        if constexpr (PAIR)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                         "r"(TMEM_COLS)
                         : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                         "r"(TMEM_COLS)
                         : "memory");
    }
    if (threadIdx.x == 0 && *abort_flag && a.status)
        atomicCAS(&a.status->code, ERR_NONE, ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_dense(const DenseArgs &args, int num_sms, cudaStream_t stream) {
    const bool pair = args.pair && !args.three;
    const int64_t bn = (args.narrow && !args.three && !pair) ? BN / 2 : BN;
    const int64_t rows = pair ? 2 * BM : BM;
    const int64_t tiles = ((args.m + rows - 1) / rows) * ((args.n + bn - 1) / bn);
    const int64_t work = args.ksplit > 1          ? tiles * args.ksplit
                         : args.tail_first >= 0 ? args.tail_first + 2 * (tiles - args.tail_first)
                                                : tiles;
    // pairs: one cluster of two CTAs per work item, at most one CTA per SM
    const int64_t units = pair ? num_sms / 2 : num_sms;
    const int grid = static_cast<int>((work < units ? work : units) * (pair ? 2 : 1));
    if (grid <= 0) return cudaSuccess;
    auto launch = [&](auto kernel, int smem, bool *attr) -> cudaError_t {
        if (!*attr) {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            *attr = true;
        }
        if (!pair) return launch_pdl(kernel, dim3(grid), dim3(THREADS), (size_t)smem, stream, args);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = (size_t)smem;
        cfg.stream = stream;
        cudaLaunchAttribute attrs[2];
        attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[0].val.programmaticStreamSerializationAllowed = 1;
        attrs[1].id = cudaLaunchAttributeClusterDimension;
        attrs[1].val.clusterDim.x = 2;
        attrs[1].val.clusterDim.y = 1;
        attrs[1].val.clusterDim.z = 1;
        cfg.attrs = attrs;
        cfg.numAttrs = 2;
        return cudaLaunchKernelEx(&cfg, kernel, args);
    };
    static bool attr_bf16 = false, attr_tf32 = false, attr_3p = false, attr_bf16x3 = false;
    static bool attr_bf16_p = false, attr_tf32_p = false, attr_bf16x3_p = false;
    cudaError_t e;
    if (args.bf16x3)
        e = pair ? launch(dense_kernel<MODE_BF16X3, true>, Cfg<MODE_BF16X3>::SMEM, &attr_bf16x3_p)
                 : launch(dense_kernel<MODE_BF16X3, false>, Cfg<MODE_BF16X3>::SMEM, &attr_bf16x3);
    else if (args.bf16)
        e = pair ? launch(dense_kernel<MODE_BF16, true>, Cfg<MODE_BF16>::SMEM, &attr_bf16_p)
                 : launch(dense_kernel<MODE_BF16, false>, Cfg<MODE_BF16>::SMEM, &attr_bf16);
    else if (args.three)
        e = launch(dense_kernel<MODE_TF32_3P, false>, Cfg<MODE_TF32_3P>::SMEM, &attr_3p);
    else
        e = pair ? launch(dense_kernel<MODE_TF32, true>, Cfg<MODE_TF32>::SMEM, &attr_tf32_p)
                 : launch(dense_kernel<MODE_TF32, false>, Cfg<MODE_TF32>::SMEM, &attr_tf32);
    return e;
}

bool encode_operand_map(CUtensorMap *map, const void *base, int64_t rows, int64_t k, int32_t fmt,
                        bool tiled, int32_t box_rows, std::string *err) {
    const bool bf16 = fmt_bf16(fmt);
    const cuuint64_t planes = static_cast<cuuint64_t>(fmt_planes(fmt));
    if (planes == 0) {
        *err = "operand is not in a planar format";
        return false;
    }
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
            *err = "cuTensorMapEncodeTiled is unavailable";
            return false;
        }
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint64_t esz = bf16 ? 2 : 4;
    if (tiled) {
        // planes of [k / kt][rows][kt]: dims (kt, rows, k / kt, planes)
        const cuuint64_t kt = ROW_BYTES / esz;
        const cuuint64_t d4[4] = {kt, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(k) / kt,
                                  planes};
        const cuuint64_t s4[3] = {kt * esz, static_cast<cuuint64_t>(rows) * kt * esz,
                                  static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(k) * esz};
        const cuuint32_t b4[4] = {static_cast<cuuint32_t>(kt), static_cast<cuuint32_t>(box_rows), 1, 1};
        const cuuint32_t e4[4] = {1, 1, 1, 1};
        CUresult r4 = encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                             4, const_cast<void *>(base), d4, s4, b4, e4,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r4 != CUDA_SUCCESS) {
            *err = "cuTensorMapEncodeTiled (4-D) failed with " + std::to_string(static_cast<int>(r4));
            return false;
        }
        return true;
    }
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows), planes};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(k) * esz,
                                   static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(k) * esz};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(ROW_BYTES / esz), static_cast<cuuint32_t>(box_rows), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                        3, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed with " + std::to_string(static_cast<int>(r));
        return false;
    }
    return true;
}

}  // namespace tn
