// The FP8 block-scaled GEMM kernel family for sm_103a: D = C + A @ B^T, E4M3 (or, for B,
// E2M1) operands, UE8M0 scales (one per row per 128-wide K block), FP32 accumulation in
// tensor memory, BF16 or FP32 out.
//
// The method is the one the DeepGEMM pages describe (README "Interface / Notes": fine-grained
// scaled FP8 GEMM with packed UE8M0 scale factors on SM100, in the NT/TN/NN/TT layouts; article
// sections 4.1 and 5.2: TMA loads of both operands, warp specialization into loader /
// tensor-core / store roles, section 7: a unified tile scheduler for L2 reuse).  The Hopper
// design on the pages promotes partial sums to CUDA-core registers to apply the scales; here
// the tcgen05 block-scaled MMA applies the UE8M0 scales in hardware and accumulates in TMEM,
// so there is no promotion.
//
// One CTA per SM, persistent over output tiles of (128 * MH) x BN, warp-specialised:
//   warp 0        TMA producer: A tile [128*MH x 128 K], B tile [BN x 128 K] (128-byte swizzle;
//                 MN-major operands in boxes of 128 MN x 128 K; E2M1 B unpacked by the TMA)
//                 into an S-stage ring.
//   warp 1 (+7)   MMA issuers, whole warps with one elected lane issuing: kind::mxf8f6f4
//                 block-scaled MMAs (K = 32) into TMEM; with MH = 2 each issuer owns one
//                 128-row half of the tile, with KS = 2 half of every stage's K steps (into its
//                 own accumulator): two instruction streams keep the tensor pipe fed.  Warp 1
//                 also owns TMEM.
//   warp 6        the scale warp: loads the packed scale words of every group of four K
//                 blocks into a 2-3-slot ring as soon as a slot frees (a group ahead of the
//                 operands) and re-lays them for tcgen05.cp.
//   warps 2-5     epilogue, one output row per thread: TMEM -> registers (BF16 rows packed in
//   (+8-11)       registers, then TMEM released) -> shared memory -> global: boxes written by
//                 TMA bulk stores (one accumulator), or 32-row slabs transposed so that warp
//                 stores are coalesced (two); with MH = 2 the second set writes the second
//                 128-row half, with MH = 1 and one accumulator the two sets split the columns.
//                 Split-K clusters reduce-scatter their partial rows between these warps.
// With MH = 1 the accumulator can be double-buffered in TMEM (ACC = 2) so that the epilogue
// of one tile overlaps the main loop of the next.  MH = 2 halves the operand bytes each SM
// ingests per multiply-add (one B tile serves 256 rows), the limit for large GEMMs.
//
// Modes (runtime): dense; M-grouped contiguous (each 128-row block takes the expert of its
// first row from m_indices, padding rows are written as +0.0); M-grouped masked (the
// per-group valid-row counts are read on the device, only valid rows are computed and
// written); K-grouped (per-group K ranges read on the device, MN-major operands, FP32 out).
// Option (runtime, MH = 1): split-K over a cluster of 2, 4 or 8 CTAs reduced through
// distributed shared memory.  Every CTA loads its own operand tiles.
//
// Every barrier wait is bounded (GemmArgs::timeout_ns).  On timeout the kernel records the
// site in the device error word, raises a CTA-wide abort flag, lets every role leave its
// loop, waits (bounded) for copies it still has in flight, frees its TMEM and returns.
#pragma once

#include <type_traits>

#include "dg_internal.h"
#include "dg_ptx.cuh"

namespace dg {

constexpr int BM = 128;       // rows per MMA: the tcgen05 M
constexpr int BK = 128;       // K per stage: one 128-byte swizzle row, one scale block
constexpr int MMA_K = 32;     // K of one kind::mxf8f6f4 MMA
constexpr int DG_ERR_TIMEOUT_CODE = 6;

template <int BN_, int STAGES_, int ACC_, int MH_ = 1, int KS_ = 1, int AR_ = 128>
struct GemmCfg {
    static constexpr int BN = BN_;
    static constexpr int STAGES = STAGES_;
    static constexpr int ACC = ACC_;
    static constexpr int MH = MH_;                      // 128-row halves of a tile
    static constexpr int TM = BM * MH;                  // rows of a tile
    // A rows loaded per stage and 128-row half: 128, or 64 for calls with at most 64 rows of A
    // (the M = 64 decode shapes), which leaves room for a deeper ring of B tiles.  The MMA still
    // reads 128 rows; rows 64-127 then come from the next buffer in shared memory and give
    // accumulator rows that are never stored or exchanged.
    static constexpr int AR = AR_;
    static_assert(AR == 128 || (AR == 64 && MH_ == 1), "64-row A stages only with one 128-row half");
    // KS = 2: two MMA issuers split each 128-K stage (K steps 0-1 and 2-3) into the two TMEM
    // accumulators, which the epilogue adds.  A block-scaled 128 x N x 32 MMA holds the tensor
    // pipe N/2 cycles, but one issuing loop (barrier wait, fence, commits per stage) keeps up
    // with no less than ~98 cycles per MMA; two issuers bring the narrow tiles of the
    // HBM-bound shapes (N = 128, 192) to ~74 and N/2 cycles.  The two accumulators then serve
    // one tile instead of alternating between tiles.
    static constexpr int KS = KS_;
    static constexpr int ISSUERS = MH * KS;
    static constexpr int ACC_ROT = KS == 2 ? 1 : ACC;   // accumulator sets rotated across tiles
    static_assert(KS == 1 || (KS == 2 && MH == 1 && ACC == 2), "K-split issuers use both accumulators of one tile");
    // warps: producer, MMA issuer, 4 epilogue, scale re-layout (MH = 1); plus a second issuer
    // and 4 more epilogue warps, one set per 128-row half (MH = 2)
    // With one 128-row half and one accumulator, the MMAs of the next tile wait for the
    // epilogue to drain TMEM: two sets of four epilogue warps then split the tile's columns.
    // So do K-split tiles wider than 128 columns: their epilogue reads two accumulators, and
    // with a whole row per thread it had registers for 16 columns per TMEM round trip only
    // (12 round trips for 192 columns, ~0.1 us each, on the critical path of every decode
    // launch); with half a row per thread it loads 32 at a time (3 round trips).
    static constexpr int EPI_COLS =
        (MH == 1 && BN_ % 64 == 0 && (ACC_ == 1 || (KS_ == 2 && BN_ > 128))) ? 2 : 1;
    static constexpr int THREADS = (MH == 2 || EPI_COLS == 2) ? 384 : (KS == 2 ? 256 : 224);
    static constexpr int EPI_THREADS = 128 * MH * EPI_COLS;
    // Warp roles.  224/256 threads: producer 0, MMA issuer 1 (and 7 with KS = 2), epilogue 2-5,
    // scale warp 6.  384 threads (two sets of epilogue warps): warpgroup 0 holds the producer
    // (0), the issuers (1, and 3 with MH = 2 or KS = 2) and the scale warp (2); warpgroups 1 and 2 the
    // epilogue warps (4-7, 8-11).  Registers are then re-split per warpgroup (setmaxnreg):
    // the launch gives every thread 168, warpgroup 0 drops to WG0_REGS and the epilogue
    // warpgroups rise to EPI_REGS, which holds a 208-column BF16 row with no spills.
    static constexpr bool WG_SPLIT = THREADS == 384;
    static constexpr uint32_t SF_WARP = WG_SPLIT ? 2u : 6u;
    static constexpr uint32_t MMA1_WARP = WG_SPLIT ? 3u : 7u;
    static constexpr uint32_t EPI0 = WG_SPLIT ? 4u : 2u;     // first warp of epilogue set 0
    static constexpr int LAUNCH_REGS = 168;                 // 65536 / 384, rounded down to 8
    static constexpr int WG0_REGS = 64;
    static constexpr int EPI_REGS = 216;
    static_assert(!WG_SPLIT || 128 * WG0_REGS + 256 * EPI_REGS <= 384 * LAUNCH_REGS,
                  "the re-split registers must fit the launch's allotment");
    static_assert(MH == 1 || MH == 2, "a tile has one or two 128-row halves");
    static_assert(BN % 16 == 0 && BN >= 32 && BN <= 256, "BN must be a multiple of 16 in [32, 256]");
    // Accumulators start on 32-column boundaries: BN columns each, ACC_STRIDE apart.
    static constexpr int ACC_STRIDE = (BN + 31) / 32 * 32;
    static constexpr int SFB_CHUNKS = (BN + 127) / 128;   // 128-row scale chunks of a B tile
    static constexpr int A_BYTES = MH * AR * BK;
    static constexpr int B_BYTES = BN * BK;
    // An MN-major B tile arrives in boxes of 128 columns (the 128-byte swizzle span): with
    // MH = 2 the stage holds whole boxes, so that BN = 224 or 192 take an MN-major B too (the
    // columns past BN are loaded and not used).  With MH = 1 only BN % 128 == 0 does.
    static constexpr int B_BOXES = (BN + 127) / 128;
    static constexpr int B_STAGE = MH == 2 ? B_BOXES * 128 * BK : B_BYTES;
    static constexpr bool B_MN_OK = MH == 2 || BN % 128 == 0;
    static constexpr int SFA_BYTES = MH * 512;
    static constexpr int SFB_BYTES = SFB_CHUNKS * 512;
    static constexpr uint32_t TX_AB = A_BYTES + B_BYTES;
    static constexpr uint32_t TX_SF = TM * 4 + BN * 4;
    // The packed scale words of a group of four K blocks travel in their own ring of SF_SLOTS
    // slots (shared memory, then TMEM).  TMEM columns: ACC x MH accumulators of BN columns,
    // then per slot and per issuer 4 columns of A scales and 4 per 128-row chunk of B scales.
    static constexpr int SF_COLS = 4 + 4 * SFB_CHUNKS;
    static constexpr int SF_SLOTS = MH == 2 ? 2 : 3;
    static constexpr int TMEM_USED = ACC * MH * ACC_STRIDE + SF_SLOTS * ISSUERS * SF_COLS;
    static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64
                                   : TMEM_USED <= 128 ? 128 : TMEM_USED <= 256 ? 256 : 512;
    static_assert(TMEM_USED <= 512, "TMEM budget exceeded");
    // Shared memory, from a 1024-byte aligned base.
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SFA = OFF_B + STAGES * B_STAGE;
    static constexpr int OFF_SFB = OFF_SFA + SF_SLOTS * SFA_BYTES;
    static constexpr int OFF_BAR = OFF_SFB + SF_SLOTS * SFB_BYTES;
    // full/empty per stage; tmem full/empty per accumulator; sf full/ready/empty per scale
    // slot; split-K reduce: 4 receive (one per TMEM lane quadrant), 8 slot-free (one per CTA
    // of the cluster), 1 unit-done.
    static constexpr int NUM_BARS = 2 * STAGES + 2 * ACC + 3 * SF_SLOTS + 13;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;  // [0] TMEM base, [1] abort flag
    static constexpr int OFF_CUM = OFF_MISC + 16;             // masked mode: m-unit prefix sums
    // Split-K receive buffer: one slot per other CTA of the cluster, each holding the (at most
    // ceil(AR / split)) rows this CTA owns, BN FP32 per row (rows padded by 16 bytes).
    static constexpr int RECV_ROW = BN * 4 + 16;
    static __host__ __device__ uint32_t off_recv(int extra_ints) {
        return (static_cast<uint32_t>(OFF_CUM + extra_ints * 4) + 15u) & ~15u;
    }
    static_assert(128 * RECV_ROW <= OFF_SFA, "split-K staging of a whole tile fits in the operand ring");
    static __host__ __device__ uint32_t recv_bytes(int split) {
        return split > 1 ? static_cast<uint32_t>((split - 1) * ((AR + split - 1) / split) * RECV_ROW) : 0u;
    }
    // Without split-K the space after the prefix sums stages the epilogue's output boxes: two
    // 1 KB buffers per epilogue warp (32 rows x 32 bytes each), the source of TMA bulk stores,
    // which need 128-byte aligned shared-memory addresses (1024 here).
    static constexpr uint32_t STAGE_OUT_BYTES = (EPI_THREADS / 32) * 2048;
    static __host__ __device__ uint32_t off_stage_out(int extra_ints) {
        return (static_cast<uint32_t>(OFF_CUM + extra_ints * 4) + 1023u) & ~1023u;
    }
    // Whether any split-K launch of this configuration fits in a CTA's shared memory (227 KB at
    // most on this architecture): if not, the kernel is built without the split-K code.
    static constexpr bool SPLITK_POSSIBLE =
        MH == 1 && EPI_COLS == 1 &&
        1024 + ((OFF_CUM + 15) & ~15) + (AR / 2) * RECV_ROW <= 227 * 1024;
    static size_t smem_bytes(int extra_ints, int split, int tma_store) {
        if (split > 1) return 1024 + off_recv(extra_ints) + recv_bytes(split);
        return 1024 + (tma_store ? off_stage_out(extra_ints) + STAGE_OUT_BYTES : off_recv(extra_ints));
    }
};

struct Unit {
    int g;          // group of A and D
    int gb;         // group of B
    int mb;         // m-tile within the group (tile rows mb*128*MH .. +128*MH)
    int nb;         // n-block
    bool zero;      // nothing to compute (padding or an empty pass): write zeros / skip
    uint32_t hmask; // MH = 2: the 128-row halves computed in this unit
    int kb_begin;   // K blocks [kb_begin, kb_end) of this unit (the CTA's split-K share, or
    int kb_end;     //   the group's K blocks in K-grouped mode)
    int koff;       // K-grouped: first K block of the group in A and B
    int kpoff;      // K-grouped: first packed scale-word row of the group
};

// Unit u of the schedule.
//  * Plain: m-tile x n-block, in raster bands of raster_n n-blocks (dense, contiguous), or
//    per group over the device-side prefix sums (masked).
//  * MH = 2, contiguous: each m-tile has two passes; the units of pass 1 follow all those of
//    pass 0.  If a tile's two halves belong to one expert, pass 0 computes both and pass 1 is
//    empty; if they belong to two experts, pass h computes half h with that half's expert.
template <int MH>
__device__ __forceinline__ Unit decode_unit(const GemmArgs& a, const int* cum, int u, int kb0, int kb1) {
    Unit t;
    t.hmask = MH == 2 ? 3u : 1u;
    t.kb_begin = kb0;
    t.kb_end = kb1;
    t.koff = 0;
    t.kpoff = 0;
    if (a.mode == MODE_K_GROUPED) {
        // Group-major; within a group, raster bands as in the dense mode.  cum[0..G] are the
        // groups' first K blocks, cum[G+1..2G+1] their first packed scale-word rows.
        const int per_group = a.num_m_units * a.num_n_blocks;
        const int g = u / per_group;
        const int r0 = u - g * per_group;
        const int per_band = a.num_m_units * a.raster_n;
        const int band = r0 / per_band;
        const int r = r0 - band * per_band;
        const int n0 = band * a.raster_n;
        const int width = min(a.raster_n, a.num_n_blocks - n0);
        t.mb = r / width;
        t.nb = n0 + (r - t.mb * width);
        t.g = g;
        t.gb = g;
        // K ranges are clipped to the call's K extent, so that group sizes summing past it
        // (a broken contract) still only read the operands' own rows.
        const int c0 = min(cum[g], a.kblocks), c1 = min(cum[g + 1], a.kblocks);
        t.koff = c0;
        t.kb_begin = 0;
        t.kb_end = c1 - c0;
        t.kpoff = cum[a.groups + 1 + g];
        t.zero = t.kb_end == 0;     // an empty group: D = C (or zeros)
        return t;
    }
    int pass = 0;
    if (MH == 2 && a.mode == MODE_CONTIGUOUS) {
        const int per_pass = a.num_units >> 1;
        if (u >= per_pass) {
            pass = 1;
            u -= per_pass;
        }
    }
    if (a.mode == MODE_MASKED) {
        // largest g with cum[g] * num_n_blocks <= u; groups with no valid rows are skipped
        int lo = 0, hi = a.groups - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (cum[mid] * a.num_n_blocks <= u) lo = mid; else hi = mid - 1;
        }
        const int local = u - cum[lo] * a.num_n_blocks;
        const int mbs = cum[lo + 1] - cum[lo];
        t.g = lo;
        t.gb = lo;
        t.mb = local % mbs;      // m-units of one B tile run side by side
        t.nb = local / mbs;
        t.zero = false;
    } else {
        const int per_band = a.num_m_units * a.raster_n;
        const int band = u / per_band;
        const int r = u - band * per_band;
        const int n0 = band * a.raster_n;
        const int width = min(a.raster_n, a.num_n_blocks - n0);
        t.mb = r / width;
        t.nb = n0 + (r - t.mb * width);
        t.g = 0;
        t.gb = 0;
        t.zero = false;
        if (a.mode == MODE_CONTIGUOUS) {
            auto expert = [&](int blk) {   // expert of 128-row block blk, -1 when none
                if (blk >= a.num_m_blocks) return -1;
                const int e = __ldg(a.m_indices + static_cast<size_t>(blk) * BM);
                return (e >= 0 && e < a.b_groups) ? e : -1;
            };
            if (MH == 2) {
                const int e0 = expert(2 * t.mb), e1 = expert(2 * t.mb + 1);
                if (e0 < 0 && e1 < 0) {
                    t.zero = pass == 0;            // all padding: pass 0 writes zeros
                    t.hmask = pass == 0 ? 3u : 0u;
                    if (pass) t.zero = true;
                } else if (e0 < 0 || e1 < 0 || e0 == e1) {
                    t.gb = e0 >= 0 ? e0 : e1;
                    t.hmask = pass == 0 ? 3u : 0u;
                    t.zero = pass != 0;            // one expert: pass 1 is empty
                } else {
                    t.gb = pass == 0 ? e0 : e1;    // two experts: one half per pass
                    t.hmask = 1u << pass;
                }
            } else {
                const int e = expert(t.mb);
                t.zero = e < 0;
                t.gb = t.zero ? 0 : e;
            }
        }
    }
    return t;
}

// Bounded wait: true when the phase completed; false after the CTA aborted or this wait
// timed out (then the error word and abort flag are set).
__device__ __forceinline__ bool wait_or_abort_body(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                                  int* err, unsigned long long timeout_ns, int site) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > timeout_ns) {
            *abort_flag = 1u;
            if (err) atomicCAS(err, 0, DG_ERR_TIMEOUT_CODE | (site << 8));
            return false;
        }
    }
}

// Same, acquiring at cluster scope: for barriers completed by other CTAs of the cluster.
__device__ __forceinline__ bool wait_cluster_or_abort_body(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                                          int* err, unsigned long long timeout_ns, int site) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait_cluster(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > timeout_ns) {
            *abort_flag = 1u;
            if (err) atomicCAS(err, 0, DG_ERR_TIMEOUT_CODE | (site << 8));
            return false;
        }
    }
}

// The bounded waits as out-of-line calls (a small main loop for the instruction cache), or
// inlined (INL): the 384-thread kernels re-split registers per warpgroup, and a call there
// would have to be compiled for every register count it is reached with.
static __device__ __noinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                                  int* err, unsigned long long timeout_ns, int site) {
    return wait_or_abort_body(bar, parity, abort_flag, err, timeout_ns, site);
}
static __device__ __noinline__ bool wait_cluster_or_abort(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                                          int* err, unsigned long long timeout_ns, int site) {
    return wait_cluster_or_abort_body(bar, parity, abort_flag, err, timeout_ns, site);
}
template <bool INL>
__device__ __forceinline__ bool wait_or_abort_t(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag, int* err,
                                                unsigned long long timeout_ns, int site) {
    if constexpr (INL) return wait_or_abort_body(bar, parity, abort_flag, err, timeout_ns, site);
    else return wait_or_abort(bar, parity, abort_flag, err, timeout_ns, site);
}
template <bool INL>
__device__ __forceinline__ bool wait_cluster_or_abort_t(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                                        int* err, unsigned long long timeout_ns, int site) {
    if constexpr (INL) return wait_cluster_or_abort_body(bar, parity, abort_flag, err, timeout_ns, site);
    else return wait_cluster_or_abort(bar, parity, abort_flag, err, timeout_ns, site);
}
template <bool INL>
__device__ __forceinline__ bool wait_fast(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag, int* err,
                                          unsigned long long timeout_ns, int site) {
    return mbar_try_wait(bar, parity) || wait_or_abort_t<INL>(bar, parity, abort_flag, err, timeout_ns, site);
}
// Whole warp: every lane waits, and the warp goes on only if every lane saw the phase complete
// (one answer for the whole warp, so its control flow stays uniform).
template <bool INL>
__device__ __forceinline__ bool wait_fast_warp(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag, int* err,
                                               unsigned long long timeout_ns, int site) {
    return __all_sync(0xffffffffu, wait_fast<INL>(bar, parity, abort_flag, err, timeout_ns, site));
}

// Re-lay one 128-row chunk of scale words (word r = row r, as TMA landed it) into the layout
// tcgen05.cp.32x128b.warpx4 expects: the 16 bytes at offset 16*i hold rows i, i+32, i+64,
// i+96.  Whole warp; in place.
__device__ __forceinline__ void relayout_sf_chunk(uint32_t* w, uint32_t lane) {
    const uint32_t v0 = w[lane], v1 = w[lane + 32], v2 = w[lane + 64], v3 = w[lane + 96];
    __syncwarp();
    reinterpret_cast<uint4*>(w)[lane] = make_uint4(v0, v1, v2, v3);
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_f32, uint32_t hi_f32) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(__uint_as_float(hi_f32)), "f"(__uint_as_float(lo_f32)));
    return r;
}

__device__ __forceinline__ void st_global_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_global_v4f(float* p, float4 v) {
    asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// Coherent load: C may alias D, which this kernel writes.
__device__ __forceinline__ float4 ld_global_v4f(const float* p) {
    float4 v;
    asm volatile("ld.global.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p)
                 : "memory");
    return v;
}

// The C values of columns [col, col + ncols) (clipped at N) of the row at `row_off`, loaded
// ahead of their use.
__device__ __forceinline__ void load_c_chunk(const GemmArgs& args, size_t row_off, int col, int N, int ncols,
                                             float4 (&cv)[8]) {
    const float* crow = args.c + row_off;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (4 * j < ncols && col + 4 * j < N) cv[j] = ld_global_v4f(crow + col + 4 * j);
}

// Stores columns [col, col + ncols) (ncols 32 or 16, clipped at N) of the output row that starts
// at element `row_off` of D, from FP32 accumulator bits r: as BF16 (round to nearest even), or
// as FP32 plus C when the call has one (cpre: C already loaded by load_c_chunk, else loaded
// here).  A zero row stores +0.0 (BF16) or C (FP32; 0 without C).
__device__ __forceinline__ void store_row_chunk(const GemmArgs& args, size_t row_off, int col, int N,
                                                const uint32_t (&r)[32], int ncols, bool zero_row,
                                                const float4* cpre = nullptr) {
    if (args.out_f32) {
        float* drow = static_cast<float*>(args.d) + row_off;
        const float* crow = args.c ? args.c + row_off : nullptr;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (4 * j < ncols && col + 4 * j < N) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (!zero_row)
                    v = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                    __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                if (crow) {
                    const float4 cv = cpre ? cpre[j] : ld_global_v4f(crow + col + 4 * j);
                    v.x += cv.x;
                    v.y += cv.y;
                    v.z += cv.z;
                    v.w += cv.w;
                }
                st_global_v4f(drow + col + 4 * j, v);
            }
        }
    } else {
        uint16_t* drow = static_cast<uint16_t*>(args.d) + row_off;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (8 * j < ncols && col + 8 * j < N) {
                uint4 v = make_uint4(0, 0, 0, 0);
                if (!zero_row) {
                    v.x = pack_bf16x2(r[8 * j + 0], r[8 * j + 1]);
                    v.y = pack_bf16x2(r[8 * j + 2], r[8 * j + 3]);
                    v.z = pack_bf16x2(r[8 * j + 4], r[8 * j + 5]);
                    v.w = pack_bf16x2(r[8 * j + 6], r[8 * j + 7]);
                }
                st_global_v4(drow + col + 8 * j, v);
            }
        }
    }
}

// A row of a tile with nothing computed (padding, an empty K group): columns [c0, c1).
__device__ __forceinline__ void store_zero_row(const GemmArgs& args, size_t row_off, int c0, int c1) {
    uint32_t none[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) none[i] = 0u;
    for (int c = c0; c < c1; c += 32) store_row_chunk(args, row_off, c, c1, none, 32, true);
}

// SPEC: SPEC_ANY, or a variant for the decode-style calls (one 128-row half; K-major
// operands, BF16 out, no C; dense or masked; E4M3 or E2M1 B) with those choices
// fixed at compile time, so that the code of the other modes is not in the kernel at all: a
// shorter instruction stream on every role's first pass, which is a visible part of a kernel
// that lives for 10-30 us.
enum : int { SPEC_ANY = 0, SPEC_DENSE = 1, SPEC_MASKED = 2, SPEC_DENSE_FP4 = 3, SPEC_MASKED_FP4 = 4 };

// 32 (or 16) accumulator columns of this thread's row into r: with K-split issuers (KS = 2)
// the sum of the two accumulators (the stage's two K halves), waited for; otherwise issued
// only (the caller waits).
template <class C, int W>
__device__ __forceinline__ void acc_ld(uint32_t taddr, uint32_t (&r)[32]) {
    static_assert(W == 32 || W == 16, "32 or 16 columns");
    if (W == 32) tmem_ld_32x32b_x32(taddr, r);
    else tmem_ld_32x32b_x16(taddr, r);
    if (C::KS == 2) {
        uint32_t r2[32];
        if (W == 32) tmem_ld_32x32b_x32(taddr + C::ACC_STRIDE, r2);
        else tmem_ld_32x32b_x16(taddr + C::ACC_STRIDE, r2);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < W; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(r2[i]));
    }
}

template <class C, int SPEC>
__global__ void __launch_bounds__(C::THREADS, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_sfa, const __grid_constant__ CUtensorMap tm_sfb,
                    const __grid_constant__ CUtensorMap tm_d, const __grid_constant__ CUtensorMap tm_d64,
                    const GemmArgs args_in) {
    GemmArgs args = args_in;
    if (SPEC != SPEC_ANY) {
        const bool dense = SPEC == SPEC_DENSE || SPEC == SPEC_DENSE_FP4;
        args.mode = dense ? MODE_DENSE : MODE_MASKED;
        if (dense) {
            args.groups = 1;
            args.b_groups = 1;
        }
        args.a_mn = 0;
        args.b_mn = 0;
        args.b_fp4 = SPEC == SPEC_DENSE_FP4 || SPEC == SPEC_MASKED_FP4;
        args.out_f32 = 0;
        args.c = nullptr;
    }
    constexpr int MH = C::MH;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const gbase = smem_raw + (base - raw);
    const uint32_t warp = threadIdx.x / 32;
    const uint32_t lane = threadIdx.x % 32;

    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(gbase + C::OFF_MISC);
    int* cum = reinterpret_cast<int*>(gbase + C::OFF_CUM);
    auto full_bar = [&](int s) { return base + C::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return base + C::OFF_BAR + 8u * (C::STAGES + s); };
    auto tfull_bar = [&](int a) { return base + C::OFF_BAR + 8u * (2 * C::STAGES + a); };
    auto tempty_bar = [&](int a) { return base + C::OFF_BAR + 8u * (2 * C::STAGES + C::ACC + a); };
    constexpr int SFB0 = 2 * C::STAGES + 2 * C::ACC;   // first scale-ring barrier
    auto sfempty_bar = [&](int j) { return base + C::OFF_BAR + 8u * (SFB0 + j); };
    auto sfready_bar = [&](int j) { return base + C::OFF_BAR + 8u * (SFB0 + C::SF_SLOTS + j); };
    auto sffull_bar = [&](int j) { return base + C::OFF_BAR + 8u * (SFB0 + 2 * C::SF_SLOTS + j); };
    auto redfull_bar = [&](int j) { return base + C::OFF_BAR + 8u * (SFB0 + 3 * C::SF_SLOTS + j); };
    auto slotfree_bar = [&](uint32_t o) { return base + C::OFF_BAR + 8u * (SFB0 + 3 * C::SF_SLOTS + 4 + o); };
    const uint32_t unitdone_bar = base + C::OFF_BAR + 8u * (SFB0 + 3 * C::SF_SLOTS + 12);
    const int split = C::SPLITK_POSSIBLE ? args.split : 1;
    const uint32_t recv_base = base + C::off_recv(extra_smem_ints(args.mode, args.groups));

    if (threadIdx.x == 0) {
        // Arrivals per phase: a stage is released by every MMA issuer; an accumulator is full
        // once every issuer committed.
        const uint32_t issuers = C::ISSUERS;
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), issuers);
        }
        for (int a = 0; a < C::ACC; ++a) {
            mbar_init(tfull_bar(a), issuers);
            mbar_init(tempty_bar(a), C::EPI_THREADS);
        }
        for (int j = 0; j < C::SF_SLOTS; ++j) {
            mbar_init(sfempty_bar(j), issuers);
            mbar_init(sfready_bar(j), 1);
            mbar_init(sffull_bar(j), 1);
        }
        for (int j = 0; j < 4; ++j) mbar_init(redfull_bar(j), 1);
        // split-K slot handshake, per unit: CTA o's slot-free barrier here takes one arrival from
        // CTA o and one from each epilogue warp of this CTA; the unit-done barrier one from each
        // epilogue warp
        for (uint32_t o = 0; o < 8; ++o) mbar_init(slotfree_bar(o), 1u + C::EPI_THREADS / 32);
        mbar_init(unitdone_bar, C::EPI_THREADS / 32);
        misc[1] = 0u;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        if (args.tma_store) {
            tma_prefetch_desc(&tm_d);
            if (C::ACC == 2 && !args.out_f32) tma_prefetch_desc(&tm_d64);
        }
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
        tma_prefetch_desc(&tm_sfa);
        tma_prefetch_desc(&tm_sfb);
    }
    if (warp == 1) {
        tmem_alloc(base + C::OFF_MISC, C::TMEM_COLS);
        tmem_relinquish();
    }
    if (args.prefetch_b && warp == 0 && lane == 0) {
        // Warm L2 with the B tiles and the scale words of this CTA's first unit (its K range of
        // one tile) while the previous kernel finishes: a prefetch reads nothing into this CTA,
        // so it is safe before the dependency wait even if that kernel writes these tensors.
        // Dense calls know their first unit here; masked calls do not (the unit map needs
        // masked_m), so they assume one m-unit per group, which names the first units' tiles
        // when groups are shallow and only warms other ones otherwise.
        const int crank0 = split > 1 ? static_cast<int>(cluster_ctarank()) : 0;
        const int u0 = split > 1 ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
        int nb = -1, mb = 0, g = 0;
        if (args.mode == MODE_DENSE) {
            if (u0 < args.num_units) {
                const int per_band = args.num_m_units * args.raster_n;
                const int band = u0 / per_band;
                const int r = u0 - band * per_band;
                const int n0 = band * args.raster_n;
                const int width = min(args.raster_n, args.num_n_blocks - n0);
                mb = r / width;
                nb = n0 + (r - mb * width);
            }
        } else if (args.mode == MODE_MASKED && u0 < args.groups * args.num_n_blocks) {
            g = u0 / args.num_n_blocks;
            nb = u0 - g * args.num_n_blocks;
        }
        if (nb >= 0) {
            const int k0 = crank0 * args.kblocks / split, k1 = (crank0 + 1) * args.kblocks / split;
            for (int kp = k0 >> 2; kp <= (k1 - 1) >> 2 && k1 > k0; ++kp) {
                tma_prefetch_l2_3d(&tm_sfb, nb * C::BN, kp, g);
                tma_prefetch_l2_3d(&tm_sfa, mb * C::TM, kp, g);
            }
            for (int kb = k0; kb < k1; ++kb) tma_prefetch_l2_3d(&tm_b, kb * BK, nb * C::BN, g);
        }
    }
    // Programmatic dependent launch: the next kernel in the stream may start launching now (its
    // CTAs still wait for this grid to complete before they touch its outputs).  Everything up
    // to each role's griddep_wait() touches only this CTA's shared and tensor memory (and L2,
    // by the prefetch), so it overlaps the previous kernel: every thread that reads or writes
    // global memory waits for that kernel first, right before its first such access.
    griddep_launch_dependents();
    if (args.mode == MODE_MASKED && warp == C::EPI0) {
        griddep_wait();
        // cum[g] = sum over g' < g of the m-units of group g' (128*MH-row tiles): each lane sums a contiguous run of groups, then an exclusive warp
        // scan over the runs.
        const int G = args.groups;
        const int per = (G + 31) / 32;
        const int g0 = min(G, static_cast<int>(lane) * per), g1 = min(G, g0 + per);
        auto units_of = [&](int g) {
            const int m = min(max(__ldg(args.masked_m + g), 0), args.rows);
            return (m + C::TM - 1) / C::TM;
        };
        int run = 0;
        for (int g = g0; g < g1; ++g) run += units_of(g);
        int incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= static_cast<uint32_t>(off)) incl += v;
        }
        int acc = incl - run;
        for (int g = g0; g < g1; ++g) {
            cum[g] = acc;
            acc += units_of(g);
        }
        if (lane == 31) cum[G] = incl;
    }
    if (args.mode == MODE_K_GROUPED && warp == C::EPI0) {
        griddep_wait();
        // cum[g] = sum over g' < g of ks[g'] / 128 (K blocks) and cum[G + 1 + g] the same sum of
        // ceil(ks[g'] / 512) (packed scale-word rows): two exclusive warp scans over runs.
        const int G = args.groups;
        const int per = (G + 31) / 32;
        const int g0 = min(G, static_cast<int>(lane) * per), g1 = min(G, g0 + per);
        auto kb_of = [&](int g) { return max(__ldg(args.ks + g), 0) / BK; };
        int run_kb = 0, run_kp = 0;
        for (int g = g0; g < g1; ++g) {
            run_kb += kb_of(g);
            run_kp += (kb_of(g) + 3) / 4;
        }
        int incl_kb = run_kb, incl_kp = run_kp;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl_kb, off);
            const int w = __shfl_up_sync(0xffffffffu, incl_kp, off);
            if (lane >= static_cast<uint32_t>(off)) {
                incl_kb += v;
                incl_kp += w;
            }
        }
        int acc_kb = incl_kb - run_kb, acc_kp = incl_kp - run_kp;
        for (int g = g0; g < g1; ++g) {
            cum[g] = acc_kb;
            cum[G + 1 + g] = acc_kp;
            acc_kb += kb_of(g);
            acc_kp += (kb_of(g) + 3) / 4;
        }
        if (lane == 31) {
            cum[G] = incl_kb;
            cum[2 * G + 1] = incl_kp;
        }
    }
    tc_fence_before_sync();
    const bool clustered = split > 1;
    // The producer needs nothing another warp prepares (except the masked and K-grouped
    // prefix sums), and it only writes its own CTA's shared memory: it arrives without
    // waiting and starts loading at once.  Everyone else waits for the barrier initialisation,
    // the TMEM address and, in a cluster, for every peer to be initialised.
    const bool early_producer = warp == 0 && args.mode != MODE_MASKED && args.mode != MODE_K_GROUPED;
    if (clustered) {
        // The early producer's warp holds thread 0, which initialised the barriers and published
        // them with fence.mbarrier_init: its arrival needs no release (measured 0.3 us sooner
        // to the first load).
        if (early_producer) cluster_arrive_relaxed();
        else cluster_arrive();
        if (!early_producer) cluster_wait();
    } else if (early_producer) {
        named_bar_arrive(1, C::THREADS);
    } else {
        named_bar_sync(1, C::THREADS);
    }
    tc_fence_after_sync();

    const uint32_t tmem_base = misc[0];
    // Split-K: the CTAs of a cluster take the same tiles; CTA `crank` covers K blocks
    // [crank * kblocks / split, (crank + 1) * kblocks / split), which may start or end inside a
    // group of four K blocks (one packed scale word): the scale path loads a word for every
    // group the range touches.
    const uint32_t crank = clustered ? cluster_ctarank() : 0u;
    const int u_first = clustered ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
    const int u_step = clustered ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);
    const int total_units = args.mode == MODE_MASKED ? cum[args.groups] * args.num_n_blocks : args.num_units;
    const int krank = split > 1 ? static_cast<int>(crank) : 0;
    const int kb0 = krank * args.kblocks / split;
    const int kb1 = (krank + 1) * args.kblocks / split;

    // 384-thread kernels: warpgroup 0 (producer, issuers, scale warp) needs few registers, the
    // epilogue warpgroups hold whole accumulator rows, so each role first moves registers from
    // the first to the others (inside its own branch, so that the compiler allocates that
    // role's code within the new count).  The host refuses to launch unless the kernel was
    // given LAUNCH_REGS per thread, so the pool always holds what the increases ask for.
    if (warp == 0) {
        if constexpr (C::WG_SPLIT) setmaxnreg_dec<C::WG0_REGS>();
        // ------------------------------------------------------------------ TMA producer
        // Like the MMA issuers: the whole warp walks the loop and waits, one elected lane arms
        // the barriers and issues the loads.
        const bool leader = elect_one_sync();
        {
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued = 0;   // stages issued in total (for the abort drain)
            bool ok = true;
            // (contiguous units read m_indices; other modes wait right before the first load,
            // after the first stage's barrier is armed)
            bool waited = args.mode == MODE_CONTIGUOUS;
            if (waited) griddep_wait();
            for (int u = u_first; ok && u < total_units; u += u_step) {
                const Unit t = decode_unit<MH>(args, cum, u, kb0, kb1);
                if (t.zero) continue;
                const int ga = args.mode == MODE_MASKED ? t.g : 0;
                for (int kb = t.kb_begin; kb < t.kb_end; ++kb) {
                    if (!wait_fast_warp<C::WG_SPLIT>(empty_bar(s), ph ^ 1u, misc + 1, args.err, args.timeout_ns,
                                                     SITE_EMPTY)) {
                        ok = false;
                        break;
                    }
                    if (static_cast<int>(issued) == args.debug_drop_stage) {
                        // Test hook: this stage's barrier is never completed, so its consumer's
                        // bounded wait runs out and the kernel takes its abort path.
                        ++issued;
                        if (++s == C::STAGES) { s = 0; ph ^= 1u; }
                        continue;
                    }
                    const int kx = (t.koff + kb) * BK;
                    const int gbz = args.mode == MODE_K_GROUPED ? 0 : t.gb;
                    const uint32_t fb = full_bar(s);
                    if (leader) {
                        // An unpacking E2M1 load counts the packed bytes it reads (half its shared-memory
                        // footprint); an MN-major B arrives in whole 128-column boxes.
                        mbar_arrive_expect_tx(fb, args.b_fp4  ? C::A_BYTES + C::B_BYTES / 2
                                                  : args.b_mn ? C::A_BYTES + C::B_BOXES * 128 * BK
                                                              : C::TX_AB);
                    }
                    if (!waited) {
                        griddep_wait();
                        waited = true;
                    }
                    if (leader) {
                        if (!args.a_mn) {
                            tma_load_3d(base + C::OFF_A + s * C::A_BYTES, &tm_a, fb, kx, t.mb * C::TM, ga);
                        } else {
                            // MN-major A: one box of 128 rows x 128 K per 128-row half, 16 KB apart
#pragma unroll
                            for (int h = 0; h < MH; ++h)
                                tma_load_3d(base + C::OFF_A + s * C::A_BYTES + h * (BM * BK), &tm_a, fb,
                                            t.mb * C::TM + h * BM, kx, ga);
                        }
                        if (C::B_MN_OK && args.b_mn) {
                            // MN-major B: one box of 128 columns x 128 K per 128 columns, 16 KB apart
                            // (the descriptor's leading-dimension stride)
#pragma unroll
                            for (int j = 0; j < C::B_BOXES; ++j)
                                tma_load_3d(base + C::OFF_B + s * C::B_STAGE + j * (128 * BK), &tm_b, fb,
                                            t.nb * C::BN + j * 128, kx, gbz);
                        } else {
                            tma_load_3d(base + C::OFF_B + s * C::B_STAGE, &tm_b, fb, kx, t.nb * C::BN, gbz);
                        }
                    }
                    ++issued;
                    if (++s == C::STAGES) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok || misc[1]) {
                // Abort: wait (bounded, short) until the loads already issued have landed.
                const uint32_t n = issued < static_cast<uint32_t>(C::STAGES) ? issued : C::STAGES;
                for (uint32_t i = 0; i < n; ++i) {
                    if (s == 0) { s = C::STAGES; ph ^= 1u; }
                    --s;
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(full_bar(s), ph) && global_timer_ns() - t0 < 100000000ull) {}
                }
            }
            __syncwarp();
        }
    } else if (warp == 1 || (C::ISSUERS == 2 && warp == C::MMA1_WARP)) {
        if constexpr (C::WG_SPLIT) setmaxnreg_dec<C::WG0_REGS>();
        // ------------------------------------------------------------------ MMA issuer(s)
        // The whole warp walks a minimal loop and waits on the barriers; one elected lane issues
        // the scale copies, MMAs and commits.  The issuing instruction stream is on the critical
        // path of the tensor pipe: with the loop's control flow and operands uniform across the
        // warp, an issuer keeps up with 128 x 128 x 32 MMAs (64 cycles each), where a loop run by
        // one lane alone took about twice that per MMA.
        // Issuer h computes the tile's 128-row half h into its own accumulator (MH = 2), or K
        // steps 2h and 2h + 1 of every stage into accumulator h (KS = 2); a unit whose half h is
        // inactive still walks every barrier (issuing no MMA) to stay in step.
        const bool leader = elect_one_sync();
        {
            if (args.mode == MODE_CONTIGUOUS) griddep_wait();   // units read m_indices
            const uint32_t h = warp == 1 ? 0u : 1u;
            int s = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t acc_ph = 0;
            int sf_slot = 0;
            uint32_t sfr_phbits = 0;   // bit j: parity of scale slot j's ready barrier
            uint32_t sfa_t = 0, sfb_t = 0;
            bool ok = true;
            bool any_commit = false;
            uint32_t last_bar = 0, last_par = 0;
            // K-major tiles advance 32 bytes (2 descriptor units) per MMA along K; MN-major tiles
            // 32 rows of 128 bytes (256 units).
            const uint32_t a_half = MH == 2 ? h * (BM * BK) : 0u;
            const uint64_t adesc0 = args.a_mn ? smem_desc_mnmajor_sw128(base + C::OFF_A + a_half)
                                              : smem_desc_kmajor_sw128(base + C::OFF_A + a_half);
            constexpr int KSTEPS = BK / MMA_K / C::KS;           // K steps of a stage per issuer
            const int k_first = C::KS == 2 ? static_cast<int>(h) * KSTEPS : 0;
            const uint64_t bdesc0 = args.b_mn ? smem_desc_mnmajor_sw128(base + C::OFF_B)
                                              : smem_desc_kmajor_sw128(base + C::OFF_B);
            const uint64_t astep = args.a_mn ? 256ull : 2ull;
            const uint64_t bstep = args.b_mn ? 256ull : 2ull;
            const uint32_t idesc0 = idesc_mxf8_e4m3(BM, C::BN, 0) | idesc_mn_major(args.a_mn, args.b_mn) |
                                    (args.b_fp4 ? idesc_b_e2m1() : 0u);
            for (int u = u_first; ok && u < total_units; u += u_step) {
                const Unit t = decode_unit<MH>(args, cum, u, kb0, kb1);
                if (t.zero) continue;
                const bool active = MH == 2 ? ((t.hmask >> h) & 1u) != 0u : (t.hmask & 1u) != 0u;
                if (!wait_fast_warp<C::WG_SPLIT>(tempty_bar(acc), acc_ph ^ 1u, misc + 1, args.err, args.timeout_ns,
                                                 SITE_TMEM_EMPTY)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>((acc * MH + h) * C::ACC_STRIDE);
                for (int kb = t.kb_begin; kb < t.kb_end; ++kb) {
                    if ((kb & 3) == 0 || kb == t.kb_begin) {
                        // First K block of a group (or of the range): copy the group's re-laid scale words from its
                        // ring slot into this issuer's TMEM slot.  (The slot's previous MMAs are
                        // complete: the producer waited for that before loading the slot.)
                        if (!wait_fast_warp<C::WG_SPLIT>(sfready_bar(sf_slot), (sfr_phbits >> sf_slot) & 1u, misc + 1,
                                                         args.err, args.timeout_ns, SITE_SF_READY)) {
                            ok = false;
                            break;
                        }
                        sfr_phbits ^= 1u << sf_slot;
                        tc_fence_after_sync();
                        sfa_t = tmem_base + static_cast<uint32_t>(C::ACC * MH * C::ACC_STRIDE +
                                                                  (sf_slot * C::ISSUERS + h) * C::SF_COLS);
                        sfb_t = sfa_t + 4u;
                        if (active && leader) {
                            tc_cp_32x128b_warpx4(sfa_t, smem_desc_sf_chunk(base + C::OFF_SFA + sf_slot * C::SFA_BYTES +
                                                                           (MH == 2 ? h : 0u) * 512));
#pragma unroll
                            for (int c = 0; c < C::SFB_CHUNKS; ++c)
                                tc_cp_32x128b_warpx4(sfb_t + 4u * c, smem_desc_sf_chunk(base + C::OFF_SFB +
                                                                                        sf_slot * C::SFB_BYTES + 512 * c));
                        }
                    }
                    if (!wait_fast_warp<C::WG_SPLIT>(full_bar(s), ph, misc + 1, args.err, args.timeout_ns, SITE_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    if (active && leader) {
                        const uint64_t adesc = adesc0 + static_cast<uint64_t>((s * C::A_BYTES) >> 4);
                        const uint64_t bdesc = bdesc0 + static_cast<uint64_t>((s * C::B_STAGE) >> 4);
                        const uint32_t sf_id = static_cast<uint32_t>(kb & 3);
                        const uint32_t idesc = idesc0 | (sf_id << 4) | (sf_id << 29);
#pragma unroll
                        for (int i = 0; i < KSTEPS; ++i) {
                            const int k = k_first + i;
                            tc_mma_mxf8f6f4(d_tmem, adesc + astep * k, bdesc + bstep * k, idesc, sfa_t, sfb_t,
                                            (kb != t.kb_begin || i != 0) ? 1u : 0u);
                        }
                    }
                    if (leader) tc_commit(empty_bar(s));
                    if ((kb & 3) == 3 || kb == t.kb_end - 1) {
                        if (leader) tc_commit(sfempty_bar(sf_slot));
                        if (++sf_slot == C::SF_SLOTS) sf_slot = 0;
                    }
                    any_commit = true;
                    last_bar = empty_bar(s);
                    last_par = ph;
                    if (++s == C::STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                if (leader) tc_commit(tfull_bar(acc));
                if (++acc == C::ACC_ROT) { acc = 0; acc_ph ^= 1u; }
            }
            if ((!ok || misc[1]) && any_commit) {
                // Abort: let the MMAs already issued finish before TMEM is freed.
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(last_bar, last_par) && global_timer_ns() - t0 < 100000000ull) {}
            }
            __syncwarp();
        }
    } else if (warp == C::SF_WARP) {
        if constexpr (C::WG_SPLIT) setmaxnreg_dec<C::WG0_REGS>();
        // ------------------------------------------------------------------ scale re-layout
        // For every group of four K blocks, in order: wait for its scale words to land in their
        // ring slot, re-lay them for tcgen05.cp, publish them to the async proxy and signal the
        // MMA issuers.  Every party uses each slot's barriers once per group, in group order, so
        // no wait is ever more than one phase from its barrier.
        // The warp also issues each group's scale loads (one elected lane), as soon as the
        // group's ring slot is free (the MMAs of the group SF_SLOTS earlier are done): a whole
        // group ahead of the A/B stages of the group, which is what hides the load latency and
        // the re-layout.
        const bool leader = elect_one_sync();
        int sf_slot = 0;
        uint32_t sff_phbits = 0;
        uint32_t sfe_phbits = 0;          // bit j: parity of scale slot j's empty barrier
        bool waited = args.mode == MODE_CONTIGUOUS;   // units read m_indices
        if (waited) griddep_wait();
        int sf_last = -1;                 // last scale slot loaded (for the abort drain)
        uint32_t sf_last_par = 0;
        bool ok = true;
        for (int u = u_first; ok && u < total_units; u += u_step) {
            const Unit t = decode_unit<MH>(args, cum, u, kb0, kb1);
            if (t.zero) continue;
            const int ga = args.mode == MODE_MASKED ? t.g : 0;
            for (int grp = t.kb_begin >> 2; grp <= (t.kb_end - 1) >> 2; ++grp) {
                const uint32_t par = ((sfe_phbits >> sf_slot) & 1u) ^ 1u;
                if (!wait_fast_warp<C::WG_SPLIT>(sfempty_bar(sf_slot), par, misc + 1, args.err, args.timeout_ns,
                                                 SITE_SF_EMPTY)) {
                    ok = false;
                    break;
                }
                const uint32_t sb = sffull_bar(sf_slot);
                if (leader) mbar_arrive_expect_tx(sb, C::TX_SF);
                if (!waited) {
                    griddep_wait();
                    waited = true;
                }
                if (leader) {
                    const int kp = t.kpoff + grp;
                    tma_load_3d(base + C::OFF_SFA + sf_slot * C::SFA_BYTES, &tm_sfa, sb, t.mb * C::TM, kp, ga);
                    tma_load_3d(base + C::OFF_SFB + sf_slot * C::SFB_BYTES, &tm_sfb, sb, t.nb * C::BN, kp,
                                args.mode == MODE_K_GROUPED ? 0 : t.gb);
                }
                sf_last = sf_slot;
                sf_last_par = (sff_phbits >> sf_slot) & 1u;
                sfe_phbits ^= 1u << sf_slot;
                if (__shfl_sync(0xffffffffu, misc[1], 0)) {   // another role gave up
                    ok = false;
                    break;
                }
                if (!wait_fast_warp<C::WG_SPLIT>(sffull_bar(sf_slot), (sff_phbits >> sf_slot) & 1u, misc + 1, args.err,
                                                 args.timeout_ns, SITE_SF_FULL)) {
                    ok = false;
                    break;
                }
                sff_phbits ^= 1u << sf_slot;
                uint32_t* sfa_w = reinterpret_cast<uint32_t*>(gbase + C::OFF_SFA + sf_slot * C::SFA_BYTES);
                uint32_t* sfb_w = reinterpret_cast<uint32_t*>(gbase + C::OFF_SFB + sf_slot * C::SFB_BYTES);
#pragma unroll
                for (int c = 0; c < MH; ++c) relayout_sf_chunk(sfa_w + 128 * c, lane);
#pragma unroll
                for (int c = 0; c < C::SFB_CHUNKS; ++c) relayout_sf_chunk(sfb_w + 128 * c, lane);
                fence_proxy_async_smem();
                __syncwarp();
                if (leader) mbar_arrive(sfready_bar(sf_slot));
                if (++sf_slot == C::SF_SLOTS) sf_slot = 0;
            }
        }
        if (leader && misc[1] && sf_last >= 0) {
            // Abort: wait (bounded, short) until the last scale load issued has landed.
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(sffull_bar(sf_last), sf_last_par) && global_timer_ns() - t0 < 100000000ull) {}
        }
    } else if (C::WG_SPLIT && C::ISSUERS == 1 && warp == 3) {
        // warpgroup 0's spare warp (one issuer): it takes part in the warpgroup's re-split only
        setmaxnreg_dec<C::WG0_REGS>();
    } else if ((warp >= C::EPI0 && warp < C::EPI0 + 4u) || ((MH == 2 || C::EPI_COLS == 2) && warp >= 8)) {
        if constexpr (C::WG_SPLIT) setmaxnreg_inc<C::EPI_REGS>();
        // ------------------------------------------------------------------ epilogue
        // Warps 2-5 write half 0 of each tile, warps 8-11 half 1 (MH = 2) or the second half of
        // the columns (EPI_COLS = 2).
        griddep_wait();
        const uint32_t q = warp & 3u;                 // the TMEM lane quadrant this warp may read
        const int my_half = (MH == 2 && warp >= 8) ? 1 : 0;
        constexpr int NCH = (C::BN + 31) / 32;        // 32-column chunks of a tile row
        const int my_cols = (C::EPI_COLS == 2 && warp >= 8) ? 1 : 0;
        const int ch_lo = my_cols * NCH / C::EPI_COLS, ch_hi = (my_cols + 1) * NCH / C::EPI_COLS;
        const bool use_c = args.out_f32 && args.c != nullptr;
        // In place (C is D): the FP32 boxes are reduce-added into D by the TMA, so C is never
        // loaded on the box path, and a tile with nothing computed leaves D as it is.
        const bool c_red = use_c && args.c_reduce != 0;
        // This warp's two 1 KB output staging buffers (no split-K: the receive region is free).
        const uint32_t ew = warp < 8 ? warp - C::EPI0 : warp - 4u;   // epilogue warp index 0..7
        const uint32_t stage_out = base + C::off_stage_out(extra_smem_ints(args.mode, args.groups)) + ew * 2048u;
        uint32_t nbox = 0;                                          // boxes this warp has stored
        const int row_in_half = static_cast<int>(q * 32 + lane);
        const int N = args.N;
        int acc = 0;
        uint32_t acc_ph = 0;
        uint32_t red_eph = 0;  // split-K: parity of the slot-free barriers
        uint32_t red_dph = 0;  // split-K: parity of the unit-done barrier
        uint32_t red_fmask = 0;  // split-K: parities of the four receive barriers
        // split-K: this warp has arrived on the final cluster barrier (on its last unit, once the
        // peers' partial rows have landed here, so that the barrier's latency overlaps the sums
        // and stores; it only waits at exit)
        bool final_arrived = false;
        bool first_red = true;   // split-K: no unit of this CTA reduced yet
        for (int u = u_first; u < total_units; u += u_step) {
            if (misc[1]) break;
            const Unit t = decode_unit<MH>(args, cum, u, kb0, kb1);
            if (t.zero && t.hmask == 0u) continue;     // an empty pass: nothing to write
            const int n0 = t.nb * C::BN;
            const int m_valid = args.mode == MODE_MASKED ? min(max(__ldg(args.masked_m + t.g), 0), args.rows)
                                                          : args.rows;
            // Row of half h of this unit for this thread, whether it is stored, and as zeros.
            auto row_of = [&](int h) { return t.mb * C::TM + h * BM + row_in_half; };
            auto row_state = [&](int row, bool& write, bool& zero_row) {
                write = row < m_valid;
                zero_row = t.zero;
                if (args.mode == MODE_CONTIGUOUS && write && !zero_row) {
                    const int e = __ldg(args.m_indices + row);
                    zero_row = (e < 0 || e >= args.b_groups);
                }
            };
            auto roff_of = [&](int row) {
                return (static_cast<size_t>(t.g) * args.rows + row) * static_cast<size_t>(N);
            };
            if (split > 1) {
                // Reduce-scatter of the cluster's partial accumulators over the tile's V valid
                // rows (rows past the call's extent are neither sent nor summed): rows
                // [o * RPO, min(V, (o + 1) * RPO)) belong to CTA o, RPO = ceil(V / split).  Every
                // lane whose valid row belongs to another CTA sends that CTA its partial row; the
                // owner's lanes wait for the other split - 1 partials, re-read their own and add
                // (on the CTA's last unit all epilogue warps share that work, see below).
                // Row r stays in TMEM lane quadrant r / 32 in every CTA, so each quadrant's warp
                // has its own receive barrier.
                // Which warps send and receive changes with V, so the slot handshake involves every
                // epilogue warp in every unit.  This CTA keeps one slot-free barrier per other CTA
                // o; its phase for unit k closes when o has read all of unit k's data (one arrival
                // from o) and every epilogue warp here has waited for the phase of unit k - 1 (one
                // local arrival each, made after that wait, so that no phase can close before all
                // the local warps have seen the one before it).  Before sending unit k a warp waits
                // for the unit k - 1 phases of all of them.  After its unit, each warp arrives on
                // the unit-done barrier and waits for the other epilogue warps there; then one
                // thread tells every other CTA that its unit's data has been read.
                const int row = row_of(0);
                bool write, zero_row;
                row_state(row, write, zero_row);
                const size_t row_off = roff_of(row);
                const uint32_t V = static_cast<uint32_t>(min(C::AR, max(0, m_valid - t.mb * BM)));
                const uint32_t usplit = static_cast<uint32_t>(split);
                const uint32_t RPO = V > 0 ? (V + usplit - 1) / usplit : 1u;
                const uint32_t RPO_CAP = (C::AR + usplit - 1) / usplit;   // rows of a receive slot
                const uint32_t r_in_tile = q * 32u + lane;
                const bool valid_row = r_in_tile < V;
                const uint32_t owner = valid_row ? r_in_tile / RPO : crank;
                const bool recv_lane = valid_row && owner == crank;
                const bool send_lane = valid_row && owner != crank;
                const uint32_t own0 = min(V, crank * RPO), own1 = min(V, own0 + RPO);   // rows this CTA owns
                const uint32_t q0 = q * 32u;
                const uint32_t ro0 = max(own0, q0), ro1 = min(own1, q0 + 32u);          // ... in this warp
                const bool warp_recv = ro0 < ro1;
                const bool warp_send = __any_sync(0xffffffffu, send_lane);
                if (t.zero) {
                    if (recv_lane && write) store_zero_row(args, row_off, n0, min(N, n0 + C::BN));
                    continue;
                }
                if (!wait_or_abort_t<C::WG_SPLIT>(tfull_bar(acc), acc_ph, misc + 1, args.err, args.timeout_ns, SITE_TMEM_FULL)) break;
                tc_fence_after_sync();
                const uint32_t t_row = tmem_base + ((q * 32u) << 16) + static_cast<uint32_t>(acc * C::ACC_STRIDE);
                // The other CTAs are done with the previous unit's receive slots.  On this CTA's
                // first unit there is no previous unit: the waits (for the phase before the
                // barriers' first) would pass at once, and are skipped, because each cluster-scope
                // acquire costs a few hundred cycles even then (measured ~0.5 us for three, on
                // the critical path of a one-unit decode GEMM).
                bool slots_free = true;
                for (uint32_t o = 0; o < usplit && slots_free && !first_red; ++o)
                    if (o != crank)
                        slots_free = wait_cluster_or_abort_t<C::WG_SPLIT>(slotfree_bar(o), red_eph ^ 1u, misc + 1, args.err,
                                                           args.timeout_ns, SITE_RED_EMPTY);
                if (!slots_free) break;
                first_red = false;
                red_eph ^= 1u;
                __syncwarp();
                if (lane == 0)
                    for (uint32_t o = 0; o < usplit; ++o)
                        if (o != crank) mbar_arrive(slotfree_bar(o));
                const bool last_unit = u + u_step >= total_units;
                // TMEM lane quadrants holding this CTA's rows (the same in every warp): the phases of
                // their receive barriers advance this unit.
                const uint32_t qr0 = own0 / 32u, qr1 = own1 > own0 ? (own1 - 1u) / 32u + 1u : qr0;
                if (last_unit) {
                    // On the CTA's last unit the operand ring is idle once the accumulator is full:
                    // every valid row's partial is staged there (tile row r at r * RECV_ROW, the
                    // receive-slot layout); each run of rows bound for one owner goes out as one
                    // bulk copy (one request instead of 16 bytes per lane and instruction; the
                    // receivers count whole padded rows), and this CTA's own rows stay for the sum.
                    const uint32_t stg = base + C::OFF_A;
                    if (__any_sync(0xffffffffu, valid_row)) {
#pragma unroll 1
                        for (int c = 0; c < C::BN / 32; ++c) {
                            uint32_t r[32];
                            acc_ld<C, 32>(t_row + 32u * c, r);
                            tmem_wait_ld();
                            if (valid_row) {
#pragma unroll
                                for (int j = 0; j < 8; ++j)
                                    st_shared_v4(stg + r_in_tile * C::RECV_ROW + 128u * c + 16u * j,
                                                 make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]));
                            }
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (warp_send && lane == 0) {
                            const uint32_t v1 = min(V, q0 + 32u);
                            for (uint32_t o = q0 / RPO; o * RPO < v1; ++o) {
                                if (o == crank) continue;
                                const uint32_t a = max(q0, o * RPO), b = min(v1, (o + 1u) * RPO);
                                const uint32_t slot = crank < o ? crank : crank - 1u;
                                bulk_copy_to_cluster(
                                    map_to_rank(recv_base + (slot * RPO_CAP + (a - o * RPO)) * C::RECV_ROW, o),
                                    stg + a * C::RECV_ROW, (b - a) * C::RECV_ROW,
                                    map_to_rank(redfull_bar(static_cast<int>(q)), o));
                            }
                        }
                    }
                    if (warp_recv && lane == ro0 - q0)      // first owned lane of the warp
                        mbar_arrive_expect_tx(redfull_bar(static_cast<int>(q)),
                                              (usplit - 1u) * (ro1 - ro0) * static_cast<uint32_t>(C::RECV_ROW));
                    tc_fence_before_sync();
                    mbar_arrive(tempty_bar(acc));
                    if (++acc == C::ACC_ROT) { acc = 0; acc_ph ^= 1u; }
                    // Every epilogue warp has staged its own rows, and the peers' rows have landed: all
                    // of them then add and store the rows this CTA owns, consecutive threads on
                    // consecutive 16-byte units of D (coalesced).  Own partial first, then the
                    // others in rank order.
                    __syncwarp();
                    if (lane == 0) mbar_arrive(unitdone_bar);
                    if (!wait_or_abort_t<C::WG_SPLIT>(unitdone_bar, red_dph, misc + 1, args.err, args.timeout_ns, SITE_RED_UNIT)) break;
                    red_dph ^= 1u;
                    bool landed = true;
                    for (uint32_t qq = qr0; qq < qr1 && landed; ++qq)
                        landed = wait_cluster_or_abort_t<C::WG_SPLIT>(redfull_bar(static_cast<int>(qq)), (red_fmask >> qq) & 1u,
                                                       misc + 1, args.err, args.timeout_ns, SITE_RED_FULL);
                    if (!landed) break;
                    for (uint32_t qq = qr0; qq < qr1; ++qq) red_fmask ^= 1u << qq;
                    // Everything the peers send here has landed, and the peers arrive only once
                    // this CTA's rows have landed there: the final barrier may count this warp.
                    // The arrival needs no release: what it guards (no CTA leaves while a peer's
                    // copy or remote arrival may still reach its shared memory) is already ordered
                    // by the receive barriers.  Every copy into or out of this CTA completes on a
                    // receive barrier that its receiver waits for before arriving, and each
                    // slot-free arrival of an earlier unit was observed by its receiver before that
                    // CTA sent the data this warp has just waited for.  (A release arrival measured
                    // ~0.2 us later.)
                    __syncwarp();
                    cluster_arrive_relaxed();
                    final_arrived = true;
                    constexpr uint32_t UPR = C::BN / 8;               // 16-byte units per row
                    const uint32_t et = (warp - C::EPI0) * 32u + lane;  // epilogue thread 0..127
                    for (uint32_t i = et; i < (own1 - own0) * UPR; i += static_cast<uint32_t>(C::EPI_THREADS)) {
                        const uint32_t rr = i / UPR, off = 32u * (i - rr * UPR);
                        uint32_t r[32];
                        const uint4 lo = ld_shared_v4(stg + (own0 + rr) * C::RECV_ROW + off);
                        const uint4 hi = ld_shared_v4(stg + (own0 + rr) * C::RECV_ROW + off + 16u);
                        float v[8] = {__uint_as_float(lo.x), __uint_as_float(lo.y), __uint_as_float(lo.z),
                                      __uint_as_float(lo.w), __uint_as_float(hi.x), __uint_as_float(hi.y),
                                      __uint_as_float(hi.z), __uint_as_float(hi.w)};
#pragma unroll
                        for (int sl = 0; sl < 7; ++sl) {
                            if (sl >= split - 1) continue;
                            const uint32_t src = recv_base + (static_cast<uint32_t>(sl) * RPO_CAP + rr) * C::RECV_ROW + off;
                            const uint4 a = ld_shared_v4(src), b = ld_shared_v4(src + 16u);
                            v[0] += __uint_as_float(a.x);
                            v[1] += __uint_as_float(a.y);
                            v[2] += __uint_as_float(a.z);
                            v[3] += __uint_as_float(a.w);
                            v[4] += __uint_as_float(b.x);
                            v[5] += __uint_as_float(b.y);
                            v[6] += __uint_as_float(b.z);
                            v[7] += __uint_as_float(b.w);
                        }
#pragma unroll
                        for (int k = 0; k < 8; ++k) r[k] = __float_as_uint(v[k]);
                        const int orow = t.mb * BM + static_cast<int>(own0 + rr);
                        bool owrite, ozero;
                        row_state(orow, owrite, ozero);
                        if (owrite) store_row_chunk(args, roff_of(orow), n0 + 8 * static_cast<int>(i - rr * UPR), N, r, 8, ozero);
                    }
                    continue;
                }
                if (warp_send) {
                    const uint32_t slot = crank < owner ? crank : crank - 1u;
                    const uint32_t dst = map_to_rank(
                        recv_base + (send_lane ? (slot * RPO_CAP + (r_in_tile - owner * RPO)) * C::RECV_ROW : 0u),
                        owner);
                    const uint32_t rbar = map_to_rank(redfull_bar(static_cast<int>(q)), owner);
#pragma unroll 1
                    for (int c = 0; c < C::BN / 32; ++c) {
                        uint32_t r[32];
                        acc_ld<C, 32>(t_row + 32u * c, r);
                        tmem_wait_ld();
                        if (send_lane) {
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                st_async_v4(dst + 128u * c + 16u * j, r[4 * j], r[4 * j + 1], r[4 * j + 2],
                                            r[4 * j + 3], rbar);
                        }
                    }
                }
                if (warp_recv) {
                    if (lane == ro0 - q0)      // first owned lane of the warp
                        mbar_arrive_expect_tx(redfull_bar(static_cast<int>(q)),
                                              (usplit - 1u) * (ro1 - ro0) * static_cast<uint32_t>(C::BN * 4));
                    __syncwarp();
                    if (!wait_cluster_or_abort_t<C::WG_SPLIT>(redfull_bar(static_cast<int>(q)), (red_fmask >> q) & 1u, misc + 1,
                                               args.err, args.timeout_ns, SITE_RED_FULL))
                        break;
                    const uint32_t src = recv_base + (recv_lane ? r_in_tile - own0 : 0u) * C::RECV_ROW;
#pragma unroll 1
                    for (int c = 0; c < C::BN / 32; ++c) {
                        uint32_t r[32];
                        acc_ld<C, 32>(t_row + 32u * c, r);
                        tmem_wait_ld();
                        if (!recv_lane) continue;
                        float v[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                        // (unrolled for up to 7 partials, so that the slots' loads are all in flight)
#pragma unroll
                        for (int sl = 0; sl < 7; ++sl) {
                            if (sl >= split - 1) continue;
                            const float4* p = reinterpret_cast<const float4*>(
                                gbase + (src - base) + static_cast<uint32_t>(sl) * RPO_CAP * C::RECV_ROW + 128u * c);
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const float4 x = p[j];
                                v[4 * j] += x.x;
                                v[4 * j + 1] += x.y;
                                v[4 * j + 2] += x.z;
                                v[4 * j + 3] += x.w;
                            }
                        }
                        if (write) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
                            store_row_chunk(args, row_off, n0 + 32 * c, N, r, 32, zero_row);
                        }
                    }
                }
                for (uint32_t qq = qr0; qq < qr1; ++qq) red_fmask ^= 1u << qq;
                tc_fence_before_sync();
                mbar_arrive(tempty_bar(acc));
                if (++acc == C::ACC_ROT) { acc = 0; acc_ph ^= 1u; }
                // Every epilogue warp is done with this unit's receive slots: tell every other CTA
                // (not after the last unit, when nothing is sent again; the final cluster barrier
                // keeps every CTA's shared memory alive until the peers' copies have landed).
                __syncwarp();
                if (lane == 0) mbar_arrive(unitdone_bar);
                if (!wait_or_abort_t<C::WG_SPLIT>(unitdone_bar, red_dph, misc + 1, args.err, args.timeout_ns, SITE_RED_UNIT)) break;
                red_dph ^= 1u;
                if (warp == C::EPI0 && lane == 0)
                    for (uint32_t rk = 0; rk < usplit; ++rk)
                        if (rk != crank) mbar_arrive_remote(map_to_rank(slotfree_bar(crank), rk));
                continue;
            }
            if (t.zero) {
                // Padding only: zeros for every row of the tile, no accumulator involved.
                if (!c_red) {
                    const int h = my_half;
                    const int row = row_of(h);
                    bool write, zero_row;
                    row_state(row, write, zero_row);
                    if (write) store_zero_row(args, roff_of(row), n0 + 32 * ch_lo, min(N, n0 + 32 * ch_hi));
                }
                continue;
            }
            float4 cv_next[8];    // FP32 with C: the next chunk's C values
            if (use_c && !c_red && ((t.hmask >> my_half) & 1u)) {
                // Ask L2 for this thread's C segment, and load its first chunk, while the tile's
                // main loop still runs.
                const int row = row_of(my_half);
                const int c0 = n0 + 32 * ch_lo, c1 = min(N, n0 + 32 * ch_hi);
                if (row < m_valid && c1 > c0) {
                    prefetch_l2(args.c + roff_of(row) + c0, static_cast<uint32_t>(c1 - c0) * 4u);
                    load_c_chunk(args, roff_of(row), c0, N, 32, cv_next);
                }
            }
            if (!wait_or_abort_t<C::WG_SPLIT>(tfull_bar(acc), acc_ph, misc + 1, args.err, args.timeout_ns, SITE_TMEM_FULL)) break;
            tc_fence_after_sync();
            {
                const int h = my_half;
                if (!((t.hmask >> h) & 1u)) goto epilogue_release;
                const int row = row_of(h);
                bool write, zero_row;
                row_state(row, write, zero_row);
                const size_t row_off = roff_of(row);
                const uint32_t t_row =
                    tmem_base + ((q * 32u) << 16) + static_cast<uint32_t>((acc * MH + h) * C::ACC_STRIDE);
                // The warp's 32 rows go out as TMA boxes unless some of them must stay untouched
                // (masked mode past masked_m[g]); rows past D's extent are clipped by the map.
                const int slab0 = row - static_cast<int>(lane);
                const bool slab_tma =
                    args.tma_store && (args.mode != MODE_MASKED || slab0 + 32 <= m_valid) && slab0 < m_valid;
                // One output box: this lane's 32 bytes of a 32-row x 32-byte box, staged in one of
                // the warp's two buffers and written by a TMA bulk store.
                auto put_box = [&](int col, uint4 w0, uint4 w1) {
                    const uint32_t buf = stage_out + (nbox & 1u) * 1024u;
                    if (nbox >= 2) {
                        // the store that last read this buffer must be done reading it
                        if (lane == 0) bulk_wait_group_read<1>();
                        __syncwarp();
                    }
                    st_shared_v4(buf + lane * 32u, w0);
                    st_shared_v4(buf + lane * 32u + 16u, w1);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (c_red) tma_reduce_add_3d(&tm_d, buf, col, slab0, t.g);
                        else if (args.d_evict_first) tma_store_3d_hint(&tm_d, buf, col, slab0, t.g, l2_policy_evict_first());
                        else tma_store_3d(&tm_d, buf, col, slab0, t.g);
                        bulk_commit_group();
                    }
                    ++nbox;
                };
                if (!args.out_f32) {
                    // BF16 out: the whole row segment goes from TMEM to registers (packed) first,
                    // so the accumulator is released before any store is issued and the stores
                    // overlap the next tile's main loop.
                    // The segment is handled in 16-column pieces (a BN that is not a multiple of 32
                    // ends in a single one).
                    constexpr int NP = C::BN / 16 / C::EPI_COLS;
                    static_assert(C::BN % (16 * C::EPI_COLS) == 0, "whole 16-column pieces per epilogue warp");
                    const int pc0 = 2 * ch_lo;                   // first piece of this thread's segment
                    uint32_t pk[NP * 8];
                    // 32 columns per TMEM load (half the round trips) where registers allow: K-split
                    // kernels load two accumulators, so those with more than 128 columns load 16 at
                    // a time (the 384-thread kernels' epilogue warps have EPI_REGS registers).
                    constexpr int LDC = ((C::THREADS <= 256 && (C::KS == 1 || C::BN <= 128)) || C::WG_SPLIT) ? 32 : 16;
                    auto load_pieces = [&](int i, auto width) {   // pieces i (and i + 1 when 32 wide)
                        uint32_t r[32];
                        const uint32_t col = t_row + 16u * static_cast<uint32_t>(pc0 + i);
                        acc_ld<C, decltype(width)::value>(col, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < decltype(width)::value / 2; ++j)
                            pk[8 * i + j] = zero_row ? 0u : pack_bf16x2(r[2 * j], r[2 * j + 1]);
                    };
                    if (LDC == 32) {
#pragma unroll
                        for (int i = 0; i < NP / 2; ++i) load_pieces(2 * i, std::integral_constant<int, 32>());
                        if (NP % 2) load_pieces(NP - 1, std::integral_constant<int, 16>());
                    } else {
#pragma unroll
                        for (int i = 0; i < NP; ++i) load_pieces(i, std::integral_constant<int, 16>());
                    }
                    tc_fence_before_sync();
                    mbar_arrive(tempty_bar(acc));
                    if (++acc == C::ACC_ROT) { acc = 0; acc_ph ^= 1u; }
                    uint16_t* drow = static_cast<uint16_t*>(args.d) + row_off;
                    // With two accumulators the stores never hold up the next tile's MMAs; they
                    // only end the CTA's last tile, where plain stores finish sooner than the
                    // chain of staged boxes.  Where the staging area exists they still go through
                    // it: each 32-row x 64-byte slab is transposed in the warp's 2 KB so that one
                    // warp store covers 8 rows x 64 contiguous bytes instead of 32 rows x 16.  The
                    // 16-byte unit j of slab row r sits at unit j ^ ((r >> 1) & 3) of the row's 64
                    // bytes, which keeps both the writes and the reads free of bank conflicts.
                    int i_direct = 0;    // first piece stored row by row
                    // On the CTA's last unit the operand ring is idle (every stage was consumed by
                    // MMAs that have completed): the warp stages its 32 rows x BN of BF16 there as
                    // 64-column boxes in the 128-byte swizzled layout (16-byte unit j of row r at
                    // unit j ^ (r mod 8): conflict-free writes) and one lane writes them out with
                    // one TMA bulk store per box.  The CTA may leave as soon as the TMA has read
                    // them, instead of after a chain of row stores.  Masked slabs that reach past
                    // masked_m keep the row stores below (rows past it stay untouched).
                    const bool last_unit_here = u + u_step >= total_units;
                    constexpr int SEG = C::BN / C::EPI_COLS;     // this warp's columns of the tile
                    if (C::ACC == 2 && args.tma_store && slab_tma && last_unit_here && SEG % 64 == 0) {
                        const uint32_t region = base + C::OFF_A + ew * static_cast<uint32_t>(32 * SEG * 2);
                        const uint32_t rsw = lane & 7u;
#pragma unroll
                        for (int b = 0; b < SEG / 64; ++b) {
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const uint32_t* p = pk + 8 * (4 * b + j / 2) + 4 * (j % 2);
                                st_shared_v4(region + static_cast<uint32_t>(b) * 4096u + lane * 128u +
                                                 16u * (static_cast<uint32_t>(j) ^ rsw),
                                             make_uint4(p[0], p[1], p[2], p[3]));
                            }
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            for (int b = 0; b < SEG / 64; ++b)
                                if (n0 + 32 * ch_lo + 64 * b < N)
                                    tma_store_3d(&tm_d64, region + static_cast<uint32_t>(b) * 4096u, n0 + 32 * ch_lo + 64 * b,
                                                 slab0, t.g);
                            bulk_commit_group();
                        }
                        ++nbox;
                        continue;   // the accumulator was released above
                    }
                    if (C::ACC == 2 && args.tma_store) {
                        uint16_t* dgrp = static_cast<uint16_t*>(args.d) +
                                         static_cast<size_t>(t.g) * args.rows * static_cast<size_t>(N);
                        const uint32_t sw = (lane >> 1) & 3u;
                        const uint32_t u = lane & 3u;
#pragma unroll
                        for (int i = 0; i + 1 < NP; i += 2) {
                            const uint32_t* p = pk + 8 * i;
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                st_shared_v4(stage_out + lane * 64u + 16u * (static_cast<uint32_t>(j) ^ sw),
                                             make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]));
                            __syncwarp();
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const uint32_t rr = 8u * k + (lane >> 2);
                                const uint4 v = ld_shared_v4(stage_out + rr * 64u + 16u * (u ^ ((rr >> 1) & 3u)));
                                const int grow = slab0 + static_cast<int>(rr);
                                const int col = n0 + 16 * (pc0 + i) + 8 * static_cast<int>(u);
                                if (grow < m_valid && col < N)
                                    st_global_v4(dgrp + static_cast<size_t>(grow) * N + col, v);
                            }
                            __syncwarp();
                        }
                        i_direct = NP & ~1;
                    }
#pragma unroll
                    for (int i = 0; i < NP; ++i) {
                        if (i < i_direct) continue;
                        const int col0 = n0 + 16 * (pc0 + i);
                        const uint32_t* p = pk + 8 * i;
                        if (slab_tma && C::ACC == 1) {
                            put_box(col0, make_uint4(p[0], p[1], p[2], p[3]), make_uint4(p[4], p[5], p[6], p[7]));
                        } else if (write) {
#pragma unroll
                            for (int j = 0; j < 2; ++j)
                                if (col0 + 8 * j < N)
                                    st_global_v4(drow + col0 + 8 * j,
                                                 make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]));
                        }
                    }
                    continue;   // the accumulator was released above
                }
                // FP32: C runs one chunk ahead in registers (the first chunk's C was loaded
                // before the wait for the accumulator), so its latency overlaps the TMEM loads
                // and the stores of the chunk before.
#pragma unroll 1
                for (int c = ch_lo; c < ch_hi; ++c) {
                    uint32_t r[32];
                    const bool half_chunk = (C::BN % 32 != 0) && (c == C::BN / 32);   // 16-column tail
                    const int ncols = half_chunk ? 16 : 32;
                    if (half_chunk) acc_ld<C, 16>(t_row + 32u * c, r);
                    else acc_ld<C, 32>(t_row + 32u * c, r);
                    float4 cv[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) cv[j] = cv_next[j];
                    if (use_c && !c_red && write && c + 1 < ch_hi)
                        load_c_chunk(args, row_off, n0 + 32 * (c + 1), N, 32, cv_next);
                    tmem_wait_ld();
                    if (!slab_tma) {
                        // (in place, C is loaded here: it was not loaded ahead)
                        if (write)
                            store_row_chunk(args, row_off, n0 + 32 * c, N, r, ncols, zero_row,
                                            (use_c && !c_red) ? cv : nullptr);
                        continue;
                    }
                    // One box = 32 rows x 32 bytes: 16 BF16 or 8 FP32 columns (fully unrolled so
                    // that r and cv stay in registers).
                    const int col0 = n0 + 32 * c;
                    if (args.out_f32) {
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            if (8 * b >= ncols) break;
                            float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
                            if (!zero_row) {
                                v0 = make_float4(__uint_as_float(r[8 * b]), __uint_as_float(r[8 * b + 1]),
                                                 __uint_as_float(r[8 * b + 2]), __uint_as_float(r[8 * b + 3]));
                                v1 = make_float4(__uint_as_float(r[8 * b + 4]), __uint_as_float(r[8 * b + 5]),
                                                 __uint_as_float(r[8 * b + 6]), __uint_as_float(r[8 * b + 7]));
                            }
                            if (use_c && !c_red && write) {
                                v0.x += cv[2 * b].x, v0.y += cv[2 * b].y, v0.z += cv[2 * b].z, v0.w += cv[2 * b].w;
                                v1.x += cv[2 * b + 1].x, v1.y += cv[2 * b + 1].y, v1.z += cv[2 * b + 1].z,
                                    v1.w += cv[2 * b + 1].w;
                            }
                            put_box(col0 + 8 * b,
                                    make_uint4(__float_as_uint(v0.x), __float_as_uint(v0.y), __float_as_uint(v0.z),
                                               __float_as_uint(v0.w)),
                                    make_uint4(__float_as_uint(v1.x), __float_as_uint(v1.y), __float_as_uint(v1.z),
                                               __float_as_uint(v1.w)));
                        }
                    } else {
#pragma unroll
                        for (int b = 0; b < 2; ++b) {
                            if (16 * b >= ncols) break;
                            uint4 w0 = make_uint4(0, 0, 0, 0), w1 = w0;
                            if (!zero_row) {
                                w0 = make_uint4(pack_bf16x2(r[16 * b + 0], r[16 * b + 1]),
                                                pack_bf16x2(r[16 * b + 2], r[16 * b + 3]),
                                                pack_bf16x2(r[16 * b + 4], r[16 * b + 5]),
                                                pack_bf16x2(r[16 * b + 6], r[16 * b + 7]));
                                w1 = make_uint4(pack_bf16x2(r[16 * b + 8], r[16 * b + 9]),
                                                pack_bf16x2(r[16 * b + 10], r[16 * b + 11]),
                                                pack_bf16x2(r[16 * b + 12], r[16 * b + 13]),
                                                pack_bf16x2(r[16 * b + 14], r[16 * b + 15]));
                            }
                            put_box(col0 + 16 * b, w0, w1);
                        }
                    }
                }
            }
        epilogue_release:
            tc_fence_before_sync();
            mbar_arrive(tempty_bar(acc));
            if (++acc == C::ACC_ROT) { acc = 0; acc_ph ^= 1u; }
        }
        // The CTA's shared memory must outlive the bulk stores' reads of it (their writes to D
        // complete on their own before the grid does).
        if (lane == 0 && nbox > 0) bulk_wait_group_read<0>();
        __syncwarp();
        if (final_arrived) {
            // the final barrier: this warp arrived early; wait with everyone else
            tc_fence_before_sync();
            if (clustered) cluster_wait();
            return;   // (TMEM is freed by warp 1 after the same barrier)
        }
    }

    tc_fence_before_sync();
    __syncwarp();
    if (clustered && early_producer) cluster_wait();   // completes the start-up barrier phase
    if (clustered) cluster_sync_all();   // no CTA leaves while a peer may still touch its memory
    else __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <class C>
cudaError_t launch_fp8_gemm(const CUtensorMap* maps, const GemmArgs& args, int grid, cudaStream_t stream) {
    const int extra = extra_smem_ints(args.mode, args.groups);
    const size_t smem = C::smem_bytes(extra, args.split, args.tma_store);
    const int cluster = args.split > 1 ? args.split : 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (args.pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    // (256-row tiles, the long prefill and MoE GEMMs, measured no faster with a variant)
    const bool plain = C::MH == 1 && !args.a_mn && !args.b_mn && !args.out_f32 && args.c == nullptr;
    const int spec = !plain                       ? SPEC_ANY
                     : args.mode == MODE_DENSE  ? (args.b_fp4 ? SPEC_DENSE_FP4 : SPEC_DENSE)
                     : args.mode == MODE_MASKED ? (args.b_fp4 ? SPEC_MASKED_FP4 : SPEC_MASKED)
                                                : SPEC_ANY;
    auto launch = [&](auto kernel) {
        return cudaLaunchKernelEx(&cfg, kernel, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], args);
    };
    constexpr bool V = C::MH == 1;   // 256-row configurations have only the general kernel
    switch (spec) {
        case SPEC_DENSE: return launch(fp8_gemm_kernel<C, V ? SPEC_DENSE : SPEC_ANY>);
        case SPEC_MASKED: return launch(fp8_gemm_kernel<C, V ? SPEC_MASKED : SPEC_ANY>);
        case SPEC_DENSE_FP4: return launch(fp8_gemm_kernel<C, V ? SPEC_DENSE_FP4 : SPEC_ANY>);
        case SPEC_MASKED_FP4: return launch(fp8_gemm_kernel<C, V ? SPEC_MASKED_FP4 : SPEC_ANY>);
        default: return launch(fp8_gemm_kernel<C, SPEC_ANY>);
    }
}

template <class C>
int max_clusters_fp8_gemm(int cluster, size_t smem) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cluster), 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fp8_gemm_kernel<C, SPEC_ANY>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

template <class C>
cudaError_t prepare_fp8_gemm(int max_smem) {
    auto prep = [&](auto kernel) {
        if (C::WG_SPLIT) {
            // The per-warpgroup register re-split draws on the registers the launch gives every
            // thread: with fewer, the epilogue's increase could never be granted.
            cudaFuncAttributes fa;
            const cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
            if (e != cudaSuccess) return e;
            if (fa.numRegs < C::LAUNCH_REGS) return cudaErrorInvalidConfiguration;
        }
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    };
    cudaError_t e = prep(fp8_gemm_kernel<C, SPEC_ANY>);
    if (e != cudaSuccess || C::MH != 1) return e;
    constexpr bool V = C::MH == 1;
    if ((e = prep(fp8_gemm_kernel<C, V ? SPEC_DENSE : SPEC_ANY>)) != cudaSuccess) return e;
    if ((e = prep(fp8_gemm_kernel<C, V ? SPEC_MASKED : SPEC_ANY>)) != cudaSuccess) return e;
    if ((e = prep(fp8_gemm_kernel<C, V ? SPEC_DENSE_FP4 : SPEC_ANY>)) != cudaSuccess) return e;
    return prep(fp8_gemm_kernel<C, V ? SPEC_MASKED_FP4 : SPEC_ANY>);
}

#define DG_DEFINE_CONFIG_AR(FN, BN_, ST_, AC_, MH_, KS_, AR_)                                             \
    const KernelConfig& FN() {                                                                             \
        using C = GemmCfg<BN_, ST_, AC_, MH_, KS_, AR_>;                                                   \
        static const KernelConfig cfg{BN_, ST_, AC_, MH_, KS_, AR_, #FN, &C::smem_bytes, &launch_fp8_gemm<C>, \
                                      &prepare_fp8_gemm<C>, &max_clusters_fp8_gemm<C>};                    \
        return cfg;                                                                                        \
    }
#define DG_DEFINE_CONFIG_KS(FN, BN_, ST_, AC_, MH_, KS_) DG_DEFINE_CONFIG_AR(FN, BN_, ST_, AC_, MH_, KS_, 128)
#define DG_DEFINE_CONFIG(FN, BN_, ST_, AC_, MH_) DG_DEFINE_CONFIG_KS(FN, BN_, ST_, AC_, MH_, 1)

}  // namespace dg
