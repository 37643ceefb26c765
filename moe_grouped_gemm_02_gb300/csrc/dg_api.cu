// The C ABI: host-side argument checks, kernel-configuration choice, TMA descriptor
// encoding and launches.  Everything here runs on the host; the arithmetic is in the
// kernels (dg_gemm_kernel.cuh, dg_pack.cu).
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "dg.h"
#include "dg_internal.h"

namespace dg {

// Set by a GEMM kernel whose barrier wait timed out; read and cleared by dg_check_device_error.
__device__ int g_device_error_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxMaskedGroups = 4096;
constexpr unsigned long long kTimeoutNs = 4000000000ull;   // 4 s per barrier wait

struct DeviceState {
    bool init = false;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    int* err_ptr = nullptr;
    int max_smem = 0;   // opt-in dynamic shared memory per block
    bool prepared = false;
    int clusters[16][7] = {};   // co-resident clusters per configuration and split 2..8 (0: unknown)
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
int g_num_sms_cap = -1;   // -1: not read from the environment yet
int g_pdl = -1;           // programmatic dependent launch: -1 unset (DG_PDL, default on), 0, 1

int pdl_enabled() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_pdl < 0) {
        const char* v = std::getenv("DG_PDL");
        g_pdl = (v && v[0] == '0') ? 0 : 1;
    }
    return g_pdl;
}

const KernelConfig* const* all_configs(int* n) {
    static const KernelConfig* cfgs[] = {&config_bn256_s4_a1(), &config_bn224_s4_a2(),
                                         &config_bn192_s5_a2(), &config_bn128_s6_a2(), &config_bn128_s4_a2(), &config_bn64_s8_a2(),
                                         &config_bn32_s8_a2(), &config_bn224_s3_m2(), &config_bn192_s3_m2(),
                                         &config_bn208_s3_m2(), &config_bn128_s5_k2(), &config_bn192_s5_k2(),
                                         &config_bn128_s8_k2_r64()};
    *n = static_cast<int>(sizeof(cfgs) / sizeof(cfgs[0]));
    return cfgs;
}

bool env_flag(const char* name) {
    const char* v = std::getenv(name);
    return v && v[0] && std::strcmp(v, "0") != 0;
}

// DG_ERR_CUDA, with the failing call printed when DG_PRINT_CONFIGS is set.
dg_status cuda_fail(const char* what, cudaError_t e) {
    if (env_flag("DG_PRINT_CONFIGS"))
        std::fprintf(stderr, "[dg] %s failed: %s\n", what, cudaGetErrorString(e));
    return DG_ERR_CUDA;
}

int sms_cap_locked() {
    if (g_num_sms_cap < 0) {
        const char* v = std::getenv("DG_NUM_SMS");
        g_num_sms_cap = v ? std::atoi(v) : 0;
        if (g_num_sms_cap < 0) g_num_sms_cap = 0;
    }
    return g_num_sms_cap;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Current device's state; initialises it (attributes, error-word address, kernel attributes)
// on first use.
dg_status current_device(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DG_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& st = g_dev[dev];
    if (!st.init) {
        cudaError_t e;
        if ((e = cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&st.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&st.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&st.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
            return cuda_fail("cudaDeviceGetAttribute", e);
        st.init = true;
    }
    if (st.cc_major != 10 || st.cc_minor != 3) return DG_ERR_UNSUPPORTED_DEVICE;
    if (!st.prepared) {
        cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&st.err_ptr), g_device_error_word);
        if (e != cudaSuccess) return cuda_fail("cudaGetSymbolAddress", e);
        int n = 0;
        const KernelConfig* const* cfgs = all_configs(&n);
        for (int i = 0; i < n; ++i)
            if ((e = cfgs[i]->prepare(st.max_smem)) != cudaSuccess) return cuda_fail("cudaFuncSetAttribute", e);
        st.prepared = true;
    }
    *out = &st;
    return DG_OK;
}

int effective_sms(const DeviceState& st) {
    std::lock_guard<std::mutex> lk(g_mu);
    const int cap = sms_cap_locked();
    return (cap > 0 && cap < st.sm_count) ? cap : st.sm_count;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int al4(int x) { return (x + 3) / 4 * 4; }

// 3-D tiled map; row_bytes is the pitch of dimension 1 (d0 elements, which for packed 4-bit
// types is d0 / 2 bytes).
bool encode_3d_pitch(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t d0, uint64_t d1,
                     uint64_t d2, uint64_t row_bytes, uint32_t b0, uint32_t b1, CUtensorMapSwizzle swz) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {row_bytes, row_bytes * d1};
    cuuint32_t box[3] = {b0, b1, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_3d(CUtensorMap* m, CUtensorMapDataType dt, uint64_t elem_bytes, const void* ptr, uint64_t d0,
               uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1, CUtensorMapSwizzle swz) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * elem_bytes, d0 * d1 * elem_bytes};
    cuuint32_t box[3] = {b0, b1, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Plan choice: a kernel configuration and a split-K factor.  The estimate, from GB300
// measurements, is waves * (K blocks per CTA * t_kb + t_tile + t_reduce).  Per K block, an SM's
// TMA moves about one 128-byte row per 2.2 cycles (A: 128 rows per half, B: BN rows) and the
// four 128 x N x 32 MMAs take N/2 cycles each, or what their issuing loop allows (see below);
// t_kb is the larger plus a quarter of the smaller.  A tile costs about 3000 cycles of fixed
// work (pipeline fill, epilogue), a split-K reduction about 5000.  Waves count tiles per
// co-resident CTA or cluster.
struct Plan {
    const KernelConfig* cfg = nullptr;
    int split = 1;
    int capacity = 0;   // co-resident CTAs (plain) or clusters (split > 1)
    int tma_store = 0;  // room for the epilogue's output staging buffers
};

int cluster_capacity(DeviceState& st, int cfg_index, const KernelConfig* c, int cluster, int slot, int split,
                     int extra_ints) {
    std::lock_guard<std::mutex> lk(g_mu);
    int& v = st.clusters[cfg_index][slot];
    if (v == 0) {
        v = c->max_clusters(cluster, c->smem_bytes(extra_ints, split, split > 1 ? 0 : 1));
        if (v <= 0) v = -1;
    }
    return v;
}

Plan choose_plan(DeviceState& st, int mode, int rows, int m_blocks_total, int N, int kblocks, int sms,
                 int extra_ints, int a_mn, int b_mn, int b_fp4, double hbm_bytes) {
    int n = 0;
    const KernelConfig* const* cfgs = all_configs(&n);
    // DG_FORCE_CONFIG=<name>, DG_FORCE_SPLIT=<1..8> pin the plan (tuning).
    const char* force_cfg = std::getenv("DG_FORCE_CONFIG");
    const char* force_split = std::getenv("DG_FORCE_SPLIT");
    const int fsplit = force_split ? std::atoi(force_split) : 0;
    Plan best;
    double best_cost = 0;
    for (int i = 0; i < n; ++i) {
        const KernelConfig* c = cfgs[i];
        if (force_cfg && std::strcmp(force_cfg, c->name) != 0) continue;
        for (int split = 1; split <= 8; ++split) {
            // Any split of 1..8 runs when forced; the planner itself takes 1, 2, 4 or 8: wider
            // odd clusters measured faster as single launches but slower back to back (64x2112:
            // split 6 8.9 vs split 4 8.5 us), where more CTAs leave fewer SMs for the next
            // kernel's early start.
            if (fsplit ? split != fsplit : (split & (split - 1)) != 0) continue;
            // 64-row A stages serve calls with at most 64 rows of K-major A (dense M, masked max_m)
            if (c->a_rows < 128 && (rows > c->a_rows || a_mn || (mode != MODE_DENSE && mode != MODE_MASKED)))
                continue;
            // MN-major B is loaded in boxes of 128 columns; K-grouped tiles have per-group K.
            if (b_mn && c->bn % 128 != 0 && c->mh != 2) continue;
            if (mode == MODE_K_GROUPED && split > 1) continue;
            // one 128-row half with one accumulator: the epilogue warps split the columns,
            // which the split-K reduction does not support
            if (split > 1 && c->mh == 1 && c->acc == 1 && c->bn % 64 == 0) continue;
            if (c->mh > 1 && split > 1) continue;
            // Masked groups are filled to an unknown, typically partial, depth: 256-row tiles
            // would mostly compute padding unless the groups are deep.
            if (c->mh > 1 && mode == MODE_MASKED && rows < 512 && !force_cfg) continue;
            if (split > 1 && (kblocks < split || c->bn % 32 != 0)) continue;
            if (c->smem_bytes(extra_ints, split, 0) > static_cast<size_t>(st.max_smem)) continue;
            const int tma_store = split == 1 && c->smem_bytes(extra_ints, 1, 1) <= static_cast<size_t>(st.max_smem);
            int cap = sms;
            if (split > 1)
                cap = std::min(cluster_capacity(st, i, c, split, split - 2, split, extra_ints), sms / split);
            if (cap <= 0) continue;
            const long long m_units = c->mh == 2 ? (m_blocks_total + 1) / 2 : m_blocks_total;
            const long long tiles = m_units * ((N + c->bn - 1) / c->bn);
            const long long waves = (tiles + cap - 1) / cap;
            const double kb_per = static_cast<double>((kblocks + split - 1) / split);
            // an MN-major B arrives in whole 128-column boxes
            const double b_rows = b_mn ? 128.0 * ((c->bn + 127) / 128) : c->bn;
            const double tma = 2.2 * (static_cast<double>(c->a_rows) * c->mh + b_rows);
            // A 128 x N x 32 MMA holds the tensor pipe N/2 cycles; the issuing loop (barrier wait and
            // fence, commits, per-stage operands) adds to that per MMA: one issuer keeps up with
            // no less than ~98 cycles, two K-split issuers ~74, two issuers of 128-row halves N/2.
            const double mma = c->mh == 2   ? 8.0 * (c->bn / 2.0)
                               : c->ks == 2 ? 4.0 * std::max(74.0, c->bn / 2.0)
                                            : 4.0 * std::max(98.0, c->bn / 2.0);
            // loads and MMAs overlap, but not perfectly: a quarter of the shorter one shows (this
            // separates tiles whose stages the loads bound alike, e.g. MN-major B tiles of 192 and
            // 224 columns, which both load 256 B columns per stage)
            const double stage = std::max(tma, mma) + 0.25 * std::min(tma, mma);
            // per tile: start and epilogue ~3000 cycles; a split-K reduction (exchange and sums
            // through distributed shared memory) ~1.7 us more once the last stage is in.  The
            // 5000 cycles were fitted when it took ~2.4 us; re-measured since, the plans they pick
            // (split 4 for the M = 64 decode shapes, none for M = 128) are still the fastest.
            const double fixed = 3000.0 + (split > 1 ? 5000.0 : 0.0);
            const double t_tile = kb_per * (stage + 20.0) + fixed;
            // however the work is spread, the operands cross HBM at ~6.2 TB/s (~3000 bytes per
            // cycle at 2.07 GHz)
            const double cost = std::max(static_cast<double>(waves) * t_tile, hbm_bytes / 3000.0 + fixed);
            // (within half a percent, the K-split issuers win: their stages go faster than
            // the estimate, which sees the larger of the load and MMA times only)
            const bool better = !best.cfg || cost < best_cost * 0.995 ||
                                (cost <= best_cost * 1.005 && c->ks > best.cfg->ks) ||
                                (cost < best_cost - 1e-9 && c->ks >= best.cfg->ks);
            if (better) {
                best.cfg = c;
                best.split = split;
                best.capacity = cap;
                best.tma_store = tma_store;
                best_cost = cost;
            }
        }
    }
    return best;
}

// One GEMM call, as the entry points describe it.
struct GemmCall {
    int mode = MODE_DENSE;
    const void* a = nullptr;
    const int32_t* sfa = nullptr;
    const void* b = nullptr;
    const int32_t* sfb = nullptr;
    void* d = nullptr;
    const float* c = nullptr;       // FP32 C (out_f32 only)
    int out_f32 = 0;
    int a_mn = 0, b_mn = 0;         // operand stored MN-major
    int b_fp4 = 0;                  // B is E2M1, two per byte
    const int32_t* m_indices = nullptr;
    const int32_t* masked_m = nullptr;
    const int32_t* ks = nullptr;    // K-grouped: K rows per group
    int groups = 1, b_groups = 1, rows = 0, N = 0, K = 0;
};

dg_status run_gemm(const GemmCall& call, void* stream) {
    const int mode = call.mode;
    const void* a = call.a;
    const int32_t* sfa = call.sfa;
    const void* b = call.b;
    const int32_t* sfb = call.sfb;
    const int32_t* m_indices = call.m_indices;
    const int32_t* masked_m = call.masked_m;
    const int groups = call.groups, b_groups = call.b_groups, rows = call.rows, N = call.N, K = call.K;
    DeviceState* st = nullptr;
    dg_status s = current_device(&st);
    if (s != DG_OK) return s;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);

    if (env_flag("DG_VALIDATE")) {
        if (cudaStreamSynchronize(cs) != cudaSuccess) return cuda_fail("cudaStreamSynchronize", cudaGetLastError());
        if (mode == MODE_CONTIGUOUS) {
            std::vector<int32_t> h(static_cast<size_t>(rows));
            if (cudaMemcpy(h.data(), m_indices, h.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
                return DG_ERR_CUDA;
            // Per 128-row block: either all -1, or a run of one expert e followed by -1s.
            // An expert's blocks are consecutive, and only the last of them may hold -1s.
            std::vector<char> seen(static_cast<size_t>(b_groups), 0);
            int prev_e = -1;
            bool prev_full = false;
            for (int blk = 0; blk < rows / 128; ++blk) {
                const int e = h[static_cast<size_t>(blk) * 128];
                if (e < -1 || e >= b_groups) return DG_ERR_CONTRACT;
                int n_valid = 0;
                bool pad = false;
                for (int r = blk * 128; r < blk * 128 + 128; ++r) {
                    const int x = h[r];
                    if (e >= 0 && x == e && !pad) ++n_valid;
                    else if (x == -1) pad = true;
                    else return DG_ERR_CONTRACT;
                }
                if (e == -1) {
                    prev_e = -1;
                    prev_full = false;
                    continue;
                }
                if (e == prev_e) {
                    if (!prev_full) return DG_ERR_CONTRACT;
                } else {
                    if (seen[e]) return DG_ERR_CONTRACT;
                    seen[e] = 1;
                }
                prev_e = e;
                prev_full = n_valid == 128;
            }
        } else if (mode == MODE_MASKED) {
            std::vector<int32_t> h(static_cast<size_t>(groups));
            if (cudaMemcpy(h.data(), masked_m, h.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
                return DG_ERR_CUDA;
            for (int g = 0; g < groups; ++g)
                if (h[g] < 0 || h[g] > rows) return DG_ERR_CONTRACT;
        } else if (mode == MODE_K_GROUPED) {
            std::vector<int32_t> h(static_cast<size_t>(groups));
            if (cudaMemcpy(h.data(), call.ks, h.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
                return DG_ERR_CUDA;
            long long sum = 0;
            for (int g = 0; g < groups; ++g) {
                if (h[g] < 0 || h[g] % 128 != 0) return DG_ERR_CONTRACT;
                sum += h[g];
            }
            if (sum != K) return DG_ERR_CONTRACT;
        }
    }

    const int sms = effective_sms(*st);
    const int m_blocks = (rows + 127) / 128;
    const int Kb = K / 128, Kp = (Kb + 3) / 4;
    const bool kgrouped = mode == MODE_K_GROUPED;
    const int extra_ints = mode == MODE_MASKED ? groups + 1 : (kgrouped ? 2 * (groups + 1) : 0);
    // K-grouped: the plan sees the mean K of a group; scale words are packed per group, at most
    // Kb / 4 + G rows in all (each group rounds its own count up).
    const int plan_kb = kgrouped ? std::max(1, (Kb + groups - 1) / groups) : Kb;
    const int kp_rows = kgrouped ? Kb / 4 + groups : Kp;
    // the operands' bytes (A as stored, B of every group, half for E2M1): what the GEMM reads
    // from HBM at least
    const double hbm_bytes = static_cast<double>(rows) * (mode == MODE_MASKED ? groups : 1) * K +
                             static_cast<double>(kgrouped ? 1 : call.b_groups) * N * K * (call.b_fp4 ? 0.5 : 1.0);
    const Plan plan = choose_plan(*st, mode, rows, m_blocks * groups, N, plan_kb, sms, extra_ints, call.a_mn,
                                  call.b_mn, call.b_fp4, hbm_bytes);
    if (!plan.cfg) return DG_ERR_SHAPE;   // nothing fits in shared memory (too many groups)
    const KernelConfig* cfg = plan.cfg;

    CUtensorMap maps[6];
    // A and D have one group per masked group; B one per expert (contiguous, masked).  K-grouped
    // operands are single [sum K, MN] matrices whose groups are K ranges.
    const int a_groups = mode == MODE_MASKED ? groups : 1;
    const int bz = kgrouped ? 1 : b_groups;
    // (A K-grouped call with sum K = 0 loads nothing: its maps get a nominal extent.)
    const int Km = K > 0 ? K : 128;
    bool ok = call.a_mn ? encode_3d(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a, rows, Km, a_groups, 128, 128,
                                    CU_TENSOR_MAP_SWIZZLE_128B)
                        : encode_3d(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a, Km, rows, a_groups, 128,
                                    cfg->a_rows * cfg->mh, CU_TENSOR_MAP_SWIZZLE_128B);
    if (call.b_fp4) {
        // E2M1 B, K-major: the TMA unpacks each 8 bytes (16 values) into a 16-byte unit, so a
        // 128-value box row fills a 128-byte swizzled row as an E4M3 row does.
        ok = ok && encode_3d_pitch(&maps[1], CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, b, Km, N, bz,
                                   static_cast<uint64_t>(Km) / 2, 128, cfg->bn, CU_TENSOR_MAP_SWIZZLE_128B);
    } else {
        ok = ok && (call.b_mn ? encode_3d(&maps[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, b, N, Km, bz, 128, 128,
                                          CU_TENSOR_MAP_SWIZZLE_128B)
                              : encode_3d(&maps[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, b, Km, N, bz, 128,
                                          cfg->bn, CU_TENSOR_MAP_SWIZZLE_128B));
    }
    ok = ok && encode_3d(&maps[2], CU_TENSOR_MAP_DATA_TYPE_INT32, 4, sfa, al4(rows), kp_rows, a_groups,
                         128 * cfg->mh, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
    ok = ok && encode_3d(&maps[3], CU_TENSOR_MAP_DATA_TYPE_INT32, 4, sfb, al4(N), kp_rows, bz, cfg->bn, 1,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    // D, for the epilogue's bulk stores: boxes of 32 rows x 32 bytes (16 BF16 or 8 FP32 values).
    const int d_groups = (mode == MODE_MASKED || kgrouped) ? groups : 1;
    if (plan.tma_store)
        ok = ok && (call.out_f32 ? encode_3d(&maps[4], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, call.d, N, rows, d_groups, 8,
                                             32, CU_TENSOR_MAP_SWIZZLE_NONE)
                                 : encode_3d(&maps[4], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, call.d, N, rows, d_groups,
                                             16, 32, CU_TENSOR_MAP_SWIZZLE_NONE));
    else
        maps[4] = maps[0];   // unused
    if (plan.tma_store && !call.out_f32)
        ok = ok && encode_3d(&maps[5], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, call.d, N, rows, d_groups, 64, 32,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    else
        maps[5] = maps[0];   // unused
    if (!ok) return cuda_fail("cuTensorMapEncodeTiled", cudaErrorInvalidValue);

    GemmArgs args{};
    args.rows = rows;
    args.N = N;
    args.K = K;
    args.mode = mode;
    args.groups = groups;
    args.b_groups = b_groups;
    args.num_m_blocks = m_blocks;
    args.num_n_blocks = (N + cfg->bn - 1) / cfg->bn;
    args.kblocks = Kb;
    args.m_indices = m_indices;
    args.masked_m = masked_m;
    args.ks = call.ks;
    args.a_mn = call.a_mn;
    args.b_mn = call.b_mn;
    args.out_f32 = call.out_f32;
    args.b_fp4 = call.b_fp4;
    args.c = call.c;
    args.d = call.d;
    args.err = st->err_ptr;
    // DG_TIMEOUT_MS shortens the bound on every barrier wait and DG_DEBUG_DROP_LOAD=n makes
    // the producer skip its n-th stage: together they let a test drive the timeout path.
    args.timeout_ns = kTimeoutNs;
    if (const char* t = std::getenv("DG_TIMEOUT_MS")) {
        const long long ms = std::atoll(t);
        if (ms > 0) args.timeout_ns = static_cast<unsigned long long>(ms) * 1000000ull;
    }
    args.debug_drop_stage = -1;
    args.pdl = pdl_enabled();
    args.tma_store = plan.tma_store;
    // An output larger than L2 cannot stay there for whoever reads it next: its stores are
    // marked evict-first, so that they do not evict the weight tiles the kernel re-reads
    // (DG_D_EVICT_FIRST=0 disables it).
    {
        const double d_bytes = static_cast<double>(rows) * N * (call.out_f32 ? 4.0 : 2.0) *
                               ((mode == MODE_MASKED || mode == MODE_K_GROUPED) ? groups : 1);
        const char* ef = std::getenv("DG_D_EVICT_FIRST");
        args.d_evict_first = (!(ef && ef[0] == '0') && d_bytes > 128.0 * 1024 * 1024) ? 1 : 0;
    }
    // D += A @ B^T in place: the epilogue's FP32 boxes are added to D by TMA reductions
    args.c_reduce = (call.out_f32 && call.c != nullptr && static_cast<const void*>(call.c) == call.d &&
                     plan.tma_store) ? 1 : 0;
    if (const char* t = std::getenv("DG_DEBUG_DROP_LOAD")) args.debug_drop_stage = std::atoi(t);
    args.num_m_units = cfg->mh == 2 ? (m_blocks + 1) / 2 : m_blocks;
    long long units_upper = static_cast<long long>(args.num_m_units) * groups * args.num_n_blocks;
    // 256-row tiles of the contiguous layout get two passes (one per expert when they straddle).
    const long long passes = (cfg->mh == 2 && mode == MODE_CONTIGUOUS) ? 2 : 1;
    if (mode == MODE_CONTIGUOUS) {
        args.raster_n = args.num_n_blocks;
    } else {
        args.raster_n = args.num_m_units >= 16 ? (args.num_n_blocks < 8 ? args.num_n_blocks : 8) : args.num_n_blocks;
    }
    args.num_units = mode == MODE_MASKED ? 0 : static_cast<int>(units_upper * passes);
    if (units_upper * passes >= (1ll << 31)) return DG_ERR_SHAPE;
    args.split = plan.split;
    // Persistent grid: one CTA (or one cluster) per co-resident slot.
    const long long slots = units_upper < plan.capacity ? units_upper : plan.capacity;
    const int grid = static_cast<int>(slots) * plan.split;
    if (env_flag("DG_PRINT_CONFIGS"))
        std::fprintf(stderr,
                     "[dg] mode=%d groups=%d rows=%d N=%d K=%d a_mn=%d b_mn=%d f32=%d -> %s (BN=%d stages=%d acc=%d "
                     "mh=%d) split=%d grid=%d raster_n=%d\n",
                     mode, groups, rows, N, K, call.a_mn, call.b_mn, call.out_f32, cfg->name, cfg->bn, cfg->stages,
                     cfg->acc, cfg->mh, plan.split, grid, args.raster_n);
    if (grid <= 0) return DG_OK;
    // Dense GEMMs whose weights fit in L2 many times over and whose grid leaves at least half
    // the SMs idle: each CTA warms L2 with its first tile's B slice and scale words before
    // waiting for the previous kernel.  The next kernel's CTAs then start on the idle SMs
    // while this one runs, and their prefetches overlap it; on a full grid the CTAs start only
    // as the previous kernel's leave, and the prefetches measured slower (queued in front of
    // the loads they were meant to warm).  DG_PREFETCH_B=0 / 1 forces it off / on.
    {
        const double b_bytes = static_cast<double>(b_groups) * N * static_cast<double>(K) * (call.b_fp4 ? 0.5 : 1.0);
        const char* pf = std::getenv("DG_PREFETCH_B");
        const bool eligible = !call.b_mn && mode == MODE_DENSE && b_bytes <= 64.0 * 1024 * 1024;
        args.prefetch_b = eligible && (pf ? pf[0] == '1' : 2 * grid <= sms) ? 1 : 0;
    }
    const cudaError_t e = cfg->launch(maps, args, grid, cs);
    return e == cudaSuccess ? DG_OK : cuda_fail("kernel launch", e);
}

dg_status check_common(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb, const void* d,
                       int N, int K) {
    if (!a || !sfa || !b || !sfb || !d) return DG_ERR_INVALID_ARG;
    if (N <= 0 || K <= 0) return DG_ERR_INVALID_ARG;
    if (K % 128 != 0 || N % 8 != 0) return DG_ERR_SHAPE;
    if (!aligned16(a) || !aligned16(sfa) || !aligned16(b) || !aligned16(sfb) || !aligned16(d))
        return DG_ERR_ALIGNMENT;
    return DG_OK;
}

// E2M1 B needs a 32-byte aligned base for the unpacking TMA, on top of the common checks.
dg_status check_fp4_b(const void* b) {
    return (reinterpret_cast<uintptr_t>(b) & 31u) ? DG_ERR_ALIGNMENT : DG_OK;
}

}  // namespace
}  // namespace dg

using namespace dg;

extern "C" {

dg_status dg_fp8_gemm_nt(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb, void* d, int M,
                         int N, int K, void* stream) {
    if (M < 0) return DG_ERR_INVALID_ARG;
    const dg_status s = check_common(a, sfa, b, sfb, d, N, K);
    if (s != DG_OK) return s;
    if (static_cast<long long>(M) * K >= (1ll << 40) || static_cast<long long>(N) * K >= (1ll << 40))
        return DG_ERR_SHAPE;
    if (M == 0) return DG_OK;
    GemmCall call;
    call.a = a, call.sfa = sfa, call.b = b, call.sfb = sfb, call.d = d;
    call.rows = M, call.N = N, call.K = K;
    return run_gemm(call, stream);
}

dg_status dg_m_grouped_fp8_gemm_nt_contiguous(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                                              void* d, const int32_t* m_indices, int M_sum, int N, int K, int G,
                                              void* stream) {
    if (M_sum < 0 || G <= 0 || !m_indices) return DG_ERR_INVALID_ARG;
    const dg_status s = check_common(a, sfa, b, sfb, d, N, K);
    if (s != DG_OK) return s;
    if (M_sum % 128 != 0) return DG_ERR_SHAPE;
    if (static_cast<long long>(M_sum) * K >= (1ll << 40) || static_cast<long long>(G) * N * K >= (1ll << 40))
        return DG_ERR_SHAPE;
    if (M_sum == 0) return DG_OK;
    GemmCall call;
    call.mode = MODE_CONTIGUOUS;
    call.a = a, call.sfa = sfa, call.b = b, call.sfb = sfb, call.d = d;
    call.m_indices = m_indices;
    call.b_groups = G, call.rows = M_sum, call.N = N, call.K = K;
    return run_gemm(call, stream);
}

dg_status dg_m_grouped_fp8_gemm_nt_masked(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                                          void* d, const int32_t* masked_m, int G, int max_m, int N, int K,
                                          void* stream) {
    if (max_m < 0 || G <= 0 || !masked_m) return DG_ERR_INVALID_ARG;
    if (G > kMaxMaskedGroups) return DG_ERR_SHAPE;
    const dg_status s = check_common(a, sfa, b, sfb, d, N, K);
    if (s != DG_OK) return s;
    if (static_cast<long long>(G) * max_m * K >= (1ll << 40) || static_cast<long long>(G) * N * K >= (1ll << 40))
        return DG_ERR_SHAPE;
    if (max_m == 0) return DG_OK;
    GemmCall call;
    call.mode = MODE_MASKED;
    call.a = a, call.sfa = sfa, call.b = b, call.sfb = sfb, call.d = d;
    call.masked_m = masked_m;
    call.groups = G, call.b_groups = G, call.rows = max_m, call.N = N, call.K = K;
    return run_gemm(call, stream);
}

dg_status dg_fp8_fp4_gemm_nt(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb, void* d, int M,
                             int N, int K, void* stream) {
    if (M < 0) return DG_ERR_INVALID_ARG;
    dg_status s = check_common(a, sfa, b, sfb, d, N, K);
    if (s != DG_OK) return s;
    if ((s = check_fp4_b(b)) != DG_OK) return s;
    if (static_cast<long long>(M) * K >= (1ll << 40) || static_cast<long long>(N) * K >= (1ll << 40))
        return DG_ERR_SHAPE;
    if (M == 0) return DG_OK;
    GemmCall call;
    call.a = a, call.sfa = sfa, call.b = b, call.sfb = sfb, call.d = d;
    call.b_fp4 = 1;
    call.rows = M, call.N = N, call.K = K;
    return run_gemm(call, stream);
}

dg_status dg_m_grouped_fp8_fp4_gemm_nt_contiguous(const void* a, const int32_t* sfa, const void* b,
                                                  const int32_t* sfb, void* d, const int32_t* m_indices, int M_sum,
                                                  int N, int K, int G, void* stream) {
    if (M_sum < 0 || G <= 0 || !m_indices) return DG_ERR_INVALID_ARG;
    dg_status s = check_common(a, sfa, b, sfb, d, N, K);
    if (s != DG_OK) return s;
    if ((s = check_fp4_b(b)) != DG_OK) return s;
    if (M_sum % 128 != 0) return DG_ERR_SHAPE;
    if (static_cast<long long>(M_sum) * K >= (1ll << 40) || static_cast<long long>(G) * N * K >= (1ll << 40))
        return DG_ERR_SHAPE;
    if (M_sum == 0) return DG_OK;
    GemmCall call;
    call.mode = MODE_CONTIGUOUS;
    call.a = a, call.sfa = sfa, call.b = b, call.sfb = sfb, call.d = d;
    call.b_fp4 = 1;
    call.m_indices = m_indices;
    call.b_groups = G, call.rows = M_sum, call.N = N, call.K = K;
    return run_gemm(call, stream);
}

dg_status dg_m_grouped_fp8_fp4_gemm_nt_masked(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                                              void* d, const int32_t* masked_m, int G, int max_m, int N, int K,
                                              void* stream) {
    if (max_m < 0 || G <= 0 || !masked_m) return DG_ERR_INVALID_ARG;
    if (G > kMaxMaskedGroups) return DG_ERR_SHAPE;
    dg_status s = check_common(a, sfa, b, sfb, d, N, K);
    if (s != DG_OK) return s;
    if ((s = check_fp4_b(b)) != DG_OK) return s;
    if (static_cast<long long>(G) * max_m * K >= (1ll << 40) || static_cast<long long>(G) * N * K >= (1ll << 40))
        return DG_ERR_SHAPE;
    if (max_m == 0) return DG_OK;
    GemmCall call;
    call.mode = MODE_MASKED;
    call.a = a, call.sfa = sfa, call.b = b, call.sfb = sfb, call.d = d;
    call.b_fp4 = 1;
    call.masked_m = masked_m;
    call.groups = G, call.b_groups = G, call.rows = max_m, call.N = N, call.K = K;
    return run_gemm(call, stream);
}

dg_status dg_fp8_gemm(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb, const float* c,
                      void* d, int M, int N, int K, int layout, int out_f32, void* stream) {
    if (M < 0 || layout < DG_LAYOUT_NT || layout > DG_LAYOUT_TT || (out_f32 != 0 && out_f32 != 1))
        return DG_ERR_INVALID_ARG;
    if (c && !out_f32) return DG_ERR_INVALID_ARG;
    const dg_status s = check_common(a, sfa, b, sfb, d, N, K);
    if (s != DG_OK) return s;
    if (c && !aligned16(c)) return DG_ERR_ALIGNMENT;
    const int a_mn = layout == DG_LAYOUT_TN || layout == DG_LAYOUT_TT;
    const int b_mn = layout == DG_LAYOUT_NN || layout == DG_LAYOUT_TN;
    // an MN-major operand's rows are M (or N) bytes long: TMA needs a 16-byte pitch
    if ((a_mn && M % 16 != 0) || (b_mn && N % 16 != 0)) return DG_ERR_SHAPE;
    if (static_cast<long long>(M) * K >= (1ll << 40) || static_cast<long long>(N) * K >= (1ll << 40))
        return DG_ERR_SHAPE;
    if (M == 0) return DG_OK;
    GemmCall call;
    call.a = a, call.sfa = sfa, call.b = b, call.sfb = sfb, call.d = d, call.c = c;
    call.out_f32 = out_f32, call.a_mn = a_mn, call.b_mn = b_mn;
    call.rows = M, call.N = N, call.K = K;
    return run_gemm(call, stream);
}

dg_status dg_k_grouped_fp8_gemm_tn_contiguous(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                                              const float* c, float* d, const int32_t* ks, int G, int M, int N,
                                              int sum_K, void* stream) {
    if (!a || !sfa || !b || !sfb || !d || !ks || G <= 0 || M < 0 || N <= 0 || sum_K < 0) return DG_ERR_INVALID_ARG;
    if (G > kMaxMaskedGroups) return DG_ERR_SHAPE;
    if (sum_K % 128 != 0 || M % 16 != 0 || N % 16 != 0) return DG_ERR_SHAPE;
    if (!aligned16(a) || !aligned16(sfa) || !aligned16(b) || !aligned16(sfb) || !aligned16(d) ||
        (c && !aligned16(c)))
        return DG_ERR_ALIGNMENT;
    if (static_cast<long long>(M) * sum_K >= (1ll << 40) || static_cast<long long>(N) * sum_K >= (1ll << 40) ||
        static_cast<long long>(G) * M * N >= (1ll << 40))
        return DG_ERR_SHAPE;
    if (M == 0) return DG_OK;
    GemmCall call;
    call.mode = MODE_K_GROUPED;
    call.a = a, call.sfa = sfa, call.b = b, call.sfb = sfb, call.d = d, call.c = c;
    call.out_f32 = 1, call.a_mn = 1, call.b_mn = 1;
    call.ks = ks;
    // sum_K == 0: every group is empty and D = C (or zeros); the kernel still runs to write it.
    call.groups = G, call.rows = M, call.N = N, call.K = sum_K;
    return run_gemm(call, stream);
}

dg_status dg_pack_sf_ue8m0(const float* sf, int32_t* out, int G, int MN, int K, int gran_mn, int gran_k,
                           void* stream) {
    if (!sf || !out || G <= 0 || MN < 0 || K <= 0) return DG_ERR_INVALID_ARG;
    if (gran_mn != 1 && gran_mn != 128) return DG_ERR_INVALID_ARG;
    if (gran_k != 128) return DG_ERR_INVALID_ARG;
    if (K % 128 != 0) return DG_ERR_SHAPE;
    if (!aligned16(out) || (reinterpret_cast<uintptr_t>(sf) & 3u)) return DG_ERR_ALIGNMENT;
    const int Kb = K / 128, Kp = (Kb + 3) / 4;
    if (Kp > 65535 || G > 65535) return DG_ERR_SHAPE;
    if (MN == 0) return DG_OK;
    DeviceState* st = nullptr;
    const dg_status s = current_device(&st);
    if (s != DG_OK) return s;
    const int MNb = (MN + gran_mn - 1) / gran_mn;
    const cudaError_t e = launch_pack_sf(sf, out, G, MN, MNb, Kb, Kp, al4(MN), gran_mn, pdl_enabled(),
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

dg_status dg_quantize_fp8_1x128(const void* x, void* q, int32_t* sf, int G, int M, int K, void* stream) {
    if (!x || !q || !sf || G <= 0 || M < 0 || K <= 0) return DG_ERR_INVALID_ARG;
    if (K % 128 != 0) return DG_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(q) || !aligned16(sf)) return DG_ERR_ALIGNMENT;
    if (M == 0) return DG_OK;
    DeviceState* st = nullptr;
    const dg_status s = current_device(&st);
    if (s != DG_OK) return s;
    const cudaError_t e = launch_quantize_fp8_1x128(x, q, sf, G, M, K, pdl_enabled(), static_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidValue) return DG_ERR_SHAPE;
    return e == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

dg_status dg_pack_sf_ue8m0_k_grouped(const float* sf, int32_t* out, const int32_t* ks, int G, int MN, int sum_K,
                                     void* stream) {
    if (!sf || !out || !ks || G <= 0 || MN < 0 || sum_K < 0) return DG_ERR_INVALID_ARG;
    if (G > kMaxMaskedGroups || sum_K % 128 != 0) return DG_ERR_SHAPE;
    if (!aligned16(out) || (reinterpret_cast<uintptr_t>(sf) & 3u)) return DG_ERR_ALIGNMENT;
    const int kb_total = sum_K / 128;
    if (kb_total / 4 + G > 65535) return DG_ERR_SHAPE;
    if (MN == 0) return DG_OK;
    DeviceState* st = nullptr;
    const dg_status s = current_device(&st);
    if (s != DG_OK) return s;
    const cudaError_t e = launch_pack_sf_k_grouped(sf, out, ks, G, MN, al4(MN), kb_total, pdl_enabled(),
                                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

int dg_get_mk_alignment_for_contiguous_layout(void) { return 128; }

int dg_get_tma_aligned_size(int mn, int elem_bytes) {
    if (mn < 0 || !(elem_bytes == 1 || elem_bytes == 2 || elem_bytes == 4 || elem_bytes == 8 || elem_bytes == 16))
        return -1;
    const int per = 16 / elem_bytes;
    return (mn + per - 1) / per * per;
}

void dg_set_num_sms(int n) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_num_sms_cap = n > 0 ? n : 0;
}

int dg_get_num_sms(void) {
    DeviceState* st = nullptr;
    if (current_device(&st) != DG_OK) {
        std::lock_guard<std::mutex> lk(g_mu);
        return sms_cap_locked();
    }
    return effective_sms(*st);
}

void dg_set_pdl(int enable) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_pdl = enable ? 1 : 0;
}

int dg_get_pdl(void) { return pdl_enabled(); }

const char* dg_status_string(dg_status s) {
    switch (s) {
        case DG_OK: return "ok";
        case DG_ERR_INVALID_ARG: return "invalid argument";
        case DG_ERR_SHAPE: return "unsupported shape";
        case DG_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
        case DG_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3";
        case DG_ERR_CUDA: return "CUDA error";
        case DG_ERR_TIMEOUT: return "kernel barrier wait timed out";
        case DG_ERR_CONTRACT: return "m_indices / masked_m violate the layout contract";
    }
    return "unknown status";
}

dg_status dg_check_device_error(void* stream) {
    DeviceState* st = nullptr;
    const dg_status s = current_device(&st);
    if (s != DG_OK) return s;
    // The word is shared by every stream on the device: wait for all of them.
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DG_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return DG_ERR_CUDA;
    int word = 0;
    if (cudaMemcpy(&word, st->err_ptr, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return DG_ERR_CUDA;
    if (word != 0) {
        const int zero = 0;
        if (cudaMemcpy(st->err_ptr, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return DG_ERR_CUDA;
        if (env_flag("DG_PRINT_CONFIGS"))
            std::fprintf(stderr, "[dg] device error word 0x%x: status %d at wait site %d\n", word, word & 0xff,
                         (word >> 8) & 0xff);
        return DG_ERR_TIMEOUT;
    }
    return DG_OK;
}

}  // extern "C"
