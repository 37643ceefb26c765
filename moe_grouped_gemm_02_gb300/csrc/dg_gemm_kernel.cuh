// The FP8 block-scaled GEMM kernel family for sm_103a: D = A @ B^T, E4M3 operands, UE8M0
// scales (one per row per 128-wide K block), FP32 accumulation in tensor memory, BF16 out.
//
// The method is the one the DeepGEMM pages describe (README "Interface / Notes": fine-grained
// scaled FP8 GEMM with packed UE8M0 scale factors on SM100; article sections 4.1 and 5.2:
// TMA loads of both operands, warp specialization into loader / tensor-core / store roles,
// section 7: a unified tile scheduler for L2 reuse).  The Hopper design on the pages promotes
// partial sums to CUDA-core registers to apply the scales; here the tcgen05 block-scaled MMA
// applies the UE8M0 scales in hardware and accumulates in TMEM, so there is no promotion.
//
// One CTA of 6 warps per SM, persistent over output tiles of 128 x BN:
//   warp 0      TMA producer: A tile [128 x 128], B tile [BN x 128] (128-byte swizzle) and
//               the packed scale words of both into an S-stage shared-memory ring.
//   warp 1      allocates TMEM; re-lays the scale words for tcgen05.cp, copies them into
//               TMEM, and one lane issues four kind::mxf8f6f4 MMAs (K = 32 each) per stage.
//   warps 2-5   epilogue: TMEM -> registers -> BF16 -> global, one output row per thread.
// The accumulator is double-buffered in TMEM when it fits (ACC = 2), so the epilogue of
// one tile overlaps the main loop of the next.
//
// Modes (runtime): dense; M-grouped contiguous (each 128-row block takes the expert of its
// first row from m_indices, padding rows are written as +0.0); M-grouped masked (the
// per-group valid-row counts are read on the device, only valid rows are computed and
// written).
//
// Every barrier wait is bounded (GemmArgs::timeout_ns).  On timeout the kernel records the
// site in the device error word, raises a CTA-wide abort flag, lets every role leave its
// loop, waits (bounded) for copies it still has in flight, frees its TMEM and returns.
#pragma once

#include "dg_internal.h"
#include "dg_ptx.cuh"

namespace dg {

constexpr int BM = 128;       // rows per tile: the tcgen05 M
constexpr int BK = 128;       // K per stage: one 128-byte swizzle row, one scale block
constexpr int MMA_K = 32;     // K of one kind::mxf8f6f4 MMA
constexpr int NUM_THREADS = 192;
constexpr int DG_ERR_TIMEOUT_CODE = 6;

template <int BN_, int STAGES_, int ACC_>
struct GemmCfg {
    static constexpr int BN = BN_;
    static constexpr int STAGES = STAGES_;
    static constexpr int ACC = ACC_;
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN must be a multiple of 32 in [32, 256]");
    static constexpr int SFB_CHUNKS = (BN + 127) / 128;   // 128-row scale chunks of a B tile
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int SFA_BYTES = 512;
    static constexpr int SFB_BYTES = SFB_CHUNKS * 512;
    static constexpr uint32_t TX_BYTES = A_BYTES + B_BYTES + BM * 4 + BN * 4;
    // TMEM columns: ACC accumulators of BN columns, then per stage 4 columns of A scales
    // and 4 per 128-row chunk of B scales.
    static constexpr int SF_COLS = 4 + 4 * SFB_CHUNKS;
    static constexpr int TMEM_USED = ACC * BN + STAGES * SF_COLS;
    static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64
                                   : TMEM_USED <= 128 ? 128 : TMEM_USED <= 256 ? 256 : 512;
    static_assert(TMEM_USED <= 512, "TMEM budget exceeded");
    // Shared memory, from a 1024-byte aligned base.
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
    static constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 2 * ACC;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;  // [0] TMEM base, [1] abort flag
    static constexpr int OFF_CUM = OFF_MISC + 16;             // masked mode: m-block prefix sums
    static size_t smem_bytes(int extra_ints) {
        return 1024 + OFF_CUM + static_cast<size_t>(extra_ints) * 4;
    }
};

struct Unit {
    int g;      // group of A and D
    int gb;     // group of B
    int mb;     // m-block within the group
    int nb;     // n-block
    bool zero;  // contiguous mode: the block is padding, write zeros only
};

__device__ __forceinline__ Unit decode_unit(const GemmArgs& a, const int* cum, int u) {
    Unit t;
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
        t.mb = local % mbs;      // m-blocks of one B tile run side by side
        t.nb = local / mbs;
        t.zero = false;
    } else {
        const int per_band = a.num_m_blocks * a.raster_n;
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
            const int e = __ldg(a.m_indices + static_cast<size_t>(t.mb) * BM);
            t.zero = (e < 0 || e >= a.b_groups);
            t.gb = t.zero ? 0 : e;
        }
    }
    return t;
}

// Bounded wait: true when the phase completed; false after the CTA aborted or this wait
// timed out (then the error word and abort flag are set).
static __device__ __noinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
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

template <class C>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_sfa, const __grid_constant__ CUtensorMap tm_sfb,
                    const GemmArgs args) {
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

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < C::ACC; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 4 * 32);
        }
        misc[1] = 0u;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
        tma_prefetch_desc(&tm_sfa);
        tma_prefetch_desc(&tm_sfb);
    }
    if (args.mode == MODE_MASKED && warp == 2) {
        // cum[g] = sum over g' < g of ceil(clamp(masked_m[g'], 0, rows) / 128): each lane sums
        // a contiguous run of groups, then an exclusive warp scan over the runs.
        const int G = args.groups;
        const int per = (G + 31) / 32;
        const int g0 = min(G, static_cast<int>(lane) * per), g1 = min(G, g0 + per);
        int run = 0;
        for (int g = g0; g < g1; ++g) {
            const int m = min(max(__ldg(args.masked_m + g), 0), args.rows);
            run += (m + BM - 1) / BM;
        }
        int incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= static_cast<uint32_t>(off)) incl += v;
        }
        int acc = incl - run;
        for (int g = g0; g < g1; ++g) {
            cum[g] = acc;
            const int m = min(max(__ldg(args.masked_m + g), 0), args.rows);
            acc += (m + BM - 1) / BM;
        }
        if (lane == 31) cum[G] = incl;
    }
    if (warp == 1) {
        tmem_alloc(base + C::OFF_MISC, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    const uint32_t tmem_base = misc[0];
    const int total_units = args.mode == MODE_MASKED ? cum[args.groups] * args.num_n_blocks : args.num_units;
    const int kblocks = args.kblocks;

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued = 0;   // stages issued in total (for the abort drain)
            bool ok = true;
            for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
                const Unit t = decode_unit(args, cum, u);
                if (t.zero) continue;
                const int ga = args.mode == MODE_MASKED ? t.g : 0;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!wait_or_abort(empty_bar(s), ph ^ 1u, misc + 1, args.err, args.timeout_ns, SITE_EMPTY)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full_bar(s);
                    mbar_arrive_expect_tx(fb, C::TX_BYTES);
                    tma_load_3d(base + C::OFF_A + s * C::A_BYTES, &tm_a, fb, kb * BK, t.mb * BM, ga);
                    tma_load_3d(base + C::OFF_B + s * C::B_BYTES, &tm_b, fb, kb * BK, t.nb * C::BN, t.gb);
                    tma_load_3d(base + C::OFF_SFA + s * C::SFA_BYTES, &tm_sfa, fb, t.mb * BM, kb >> 2, ga);
                    tma_load_3d(base + C::OFF_SFB + s * C::SFB_BYTES, &tm_sfb, fb, t.nb * C::BN, kb >> 2, t.gb);
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
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        int s = 0;
        uint32_t ph = 0;
        int acc = 0;
        uint32_t acc_ph = 0;
        bool ok = true;
        bool any_commit = false;
        uint32_t last_bar = 0, last_par = 0;
        for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
            const Unit t = decode_unit(args, cum, u);
            if (t.zero) continue;
            if (!wait_or_abort(tempty_bar(acc), acc_ph ^ 1u, misc + 1, args.err, args.timeout_ns, SITE_TMEM_EMPTY)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::BN);
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!wait_or_abort(full_bar(s), ph, misc + 1, args.err, args.timeout_ns, SITE_FULL)) {
                    ok = false;
                    break;
                }
                uint32_t* sfa_w = reinterpret_cast<uint32_t*>(gbase + C::OFF_SFA + s * C::SFA_BYTES);
                uint32_t* sfb_w = reinterpret_cast<uint32_t*>(gbase + C::OFF_SFB + s * C::SFB_BYTES);
                relayout_sf_chunk(sfa_w, lane);
#pragma unroll
                for (int c = 0; c < C::SFB_CHUNKS; ++c) relayout_sf_chunk(sfb_w + 128 * c, lane);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tc_fence_after_sync();
                    const uint32_t sfa_t = tmem_base + static_cast<uint32_t>(C::ACC * C::BN + s * C::SF_COLS);
                    const uint32_t sfb_t = sfa_t + 4u;
                    tc_cp_32x128b_warpx4(sfa_t, smem_desc_sf_chunk(base + C::OFF_SFA + s * C::SFA_BYTES));
#pragma unroll
                    for (int c = 0; c < C::SFB_CHUNKS; ++c)
                        tc_cp_32x128b_warpx4(sfb_t + 4u * c,
                                             smem_desc_sf_chunk(base + C::OFF_SFB + s * C::SFB_BYTES + 512 * c));
                    const uint64_t adesc = smem_desc_kmajor_sw128(base + C::OFF_A + s * C::A_BYTES);
                    const uint64_t bdesc = smem_desc_kmajor_sw128(base + C::OFF_B + s * C::B_BYTES);
                    const uint32_t idesc = idesc_mxf8_e4m3(BM, C::BN, static_cast<uint32_t>(kb & 3));
#pragma unroll
                    for (int k = 0; k < BK / MMA_K; ++k)
                        tc_mma_mxf8f6f4(d_tmem, adesc + 2ull * k, bdesc + 2ull * k, idesc, sfa_t, sfb_t,
                                        (kb | k) != 0 ? 1u : 0u);
                    tc_commit(empty_bar(s));
                }
                __syncwarp();
                any_commit = true;
                last_bar = empty_bar(s);
                last_par = ph;
                if (++s == C::STAGES) { s = 0; ph ^= 1u; }
            }
            if (!ok) break;
            if (lane == 0) tc_commit(tfull_bar(acc));
            __syncwarp();
            if (++acc == C::ACC) { acc = 0; acc_ph ^= 1u; }
        }
        if ((!ok || misc[1]) && any_commit) {
            // Abort: let the MMAs already issued finish before TMEM is freed.
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(last_bar, last_par) && global_timer_ns() - t0 < 100000000ull) {}
        }
    } else {
        // ------------------------------------------------------------------ epilogue
        const uint32_t q = warp & 3u;                 // the TMEM lane quadrant this warp may read
        const int row_in_tile = static_cast<int>(q * 32 + lane);
        const int N = args.N;
        int acc = 0;
        uint32_t acc_ph = 0;
        for (int u = blockIdx.x; u < total_units; u += gridDim.x) {
            if (misc[1]) break;
            const Unit t = decode_unit(args, cum, u);
            const int row = t.mb * BM + row_in_tile;
            const int n0 = t.nb * C::BN;
            bool write = row < args.rows;
            bool zero_row = t.zero;
            if (args.mode == MODE_CONTIGUOUS && write && !zero_row) {
                const int e = __ldg(args.m_indices + row);
                zero_row = (e < 0 || e >= args.b_groups);
            } else if (args.mode == MODE_MASKED) {
                const int m = min(max(__ldg(args.masked_m + t.g), 0), args.rows);
                write = row < m;
            }
            uint16_t* drow = args.d + (static_cast<size_t>(t.g) * args.rows + row) * static_cast<size_t>(N);
            if (t.zero) {
                if (write)
                    for (int c = n0; c < min(N, n0 + C::BN); c += 8) st_global_v4(drow + c, make_uint4(0, 0, 0, 0));
                continue;
            }
            if (!wait_or_abort(tfull_bar(acc), acc_ph, misc + 1, args.err, args.timeout_ns, SITE_TMEM_FULL)) break;
            tc_fence_after_sync();
            const uint32_t t_row = tmem_base + ((q * 32u) << 16) + static_cast<uint32_t>(acc * C::BN);
#pragma unroll 1
            for (int c = 0; c < C::BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_row + 32u * c, r);
                tmem_wait_ld();
                if (write) {
                    const int col = n0 + 32 * c;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (col + 8 * j < N) {
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
            tc_fence_before_sync();
            mbar_arrive(tempty_bar(acc));
            if (++acc == C::ACC) { acc = 0; acc_ph ^= 1u; }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <class C>
cudaError_t launch_fp8_gemm(const CUtensorMap* maps, const GemmArgs& args, int grid, cudaStream_t stream) {
    const int extra = args.mode == MODE_MASKED ? args.groups + 1 : 0;
    const size_t smem = C::smem_bytes(extra);
    fp8_gemm_kernel<C><<<grid, NUM_THREADS, smem, stream>>>(maps[0], maps[1], maps[2], maps[3], args);
    return cudaGetLastError();
}

template <class C>
cudaError_t prepare_fp8_gemm(int max_smem) {
    return cudaFuncSetAttribute(fp8_gemm_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

#define DG_DEFINE_CONFIG(FN, BN_, ST_, AC_)                                                          \
    const KernelConfig& FN() {                                                                        \
        using C = GemmCfg<BN_, ST_, AC_>;                                                             \
        static const KernelConfig cfg{BN_, ST_, AC_, #FN, &C::smem_bytes, &launch_fp8_gemm<C>,        \
                                      &prepare_fp8_gemm<C>};                                          \
        return cfg;                                                                                   \
    }

}  // namespace dg
