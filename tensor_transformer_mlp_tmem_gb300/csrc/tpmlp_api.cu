// The C ABI of the tensor-parallel MLP library (declared in include/tpmlp.h): argument
// checks, buffers, tensor-map encoding and kernel launches. No C++ exception and no abort
// crosses this boundary: every entry point returns a tpmlp_status.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "tpmlp.h"
#include "tpmlp_gemm.cuh"
#include "tpmlp_gemm_2sm.cuh"
#include "tpmlp_norm.cuh"
#include "tpmlp_reduce.cuh"
#include "tpmlp_pack.cuh"
#include "tpmlp_plan.h"

// Row chunks of tpmlp_forward_host's pipeline at most (sizes the context's event arrays).
#ifndef TPMLP_HOST_CHUNKS_MAX
#define TPMLP_HOST_CHUNKS_MAX 4
#endif
static_assert(TPMLP_HOST_CHUNKS_MAX >= 1 && TPMLP_HOST_CHUNKS_MAX <= 16, "host chunk limit");

struct tpmlp_ctx {
    int device = -1;
    int num_sms = 0;
    int64_t H = 0, F = 0, f = 0;
    int32_t k = 0;
    uint32_t flags = 0;
    int bn1 = 0, bn2 = 0;  // output tile widths of GEMM1 / GEMM2

    uint16_t* W1p = nullptr;  // [k][f][H]  (gated: [k][2f][H])
    uint16_t* W2p = nullptr;  // [k][H][f]
    float* b1 = nullptr;      // [F]        (gated: [2F])
    float* b2 = nullptr;      // [H]
    bool packed = false;
    CUtensorMap tmW1{}, tmW2{};            // B boxes for the single-SM kernel (BN rows)
    CUtensorMap tmW1_pair{}, tmW2_pair{};  // B boxes for the CTA-pair kernel (128 rows)
    bool pair1 = false, pair2 = false;     // GEMM1 / GEMM2 run on CTA pairs
    int kind = 0;        // 0: MLP block; 1: column-parallel linear; 2: row-parallel linear
    bool gated = false;  // SwiGLU block: W1p holds gate and up rows interleaved
    int gate_block = 0;  // G: gate/up interleave block (output columns per half-tile)

    uint16_t* Y = nullptr;  // [y_rows][F] intermediate activations
    int64_t y_rows = 0;
    void* Xs = nullptr;  // staging for tpmlp_forward_host
    void* Zs = nullptr;
    int64_t stage_rows = 0;
    cudaStream_t s_in = nullptr, s_out = nullptr;  // its copy streams (created on first use)
    cudaEvent_t host_ev[TPMLP_HOST_CHUNKS_MAX + 1] = {}, in_ev[TPMLP_HOST_CHUNKS_MAX] = {},
                out_ev[TPMLP_HOST_CHUNKS_MAX] = {};
    // row chunks of the last tpmlp_forward_host call (re-planned when M changes)
    int64_t plan_M = -1;
    int plan_n = 0;
    int64_t plan_rows[TPMLP_HOST_CHUNKS_MAX] = {};
    // tpmlp_forward_host_async: two staging slots used in turn, so that a call's copies in and
    // out overlap the kernels of the calls before and after it
    void* Xa[2] = {};
    void* Za[2] = {};
    int64_t async_rows = 0;
    cudaEvent_t a_in[2] = {}, a_xfree[2] = {}, a_zready[2] = {}, a_zfree[2] = {};
    bool a_used[2] = {};
    uint32_t a_calls = 0;

    // activation tensor maps of the last call (re-encoded only when pointer or rows change)
    const void* x_map_ptr = nullptr;
    int64_t x_map_rows = -1;
    CUtensorMap tmX{};
    const void* y_map_ptr = nullptr;
    int64_t y_map_rows = -1;
    CUtensorMap tmY{};

    // LayerNorm in front of the block (tpmlp_set_layernorm / tpmlp_block_forward)
    float* ln_gamma = nullptr;  // [H] fp32
    float* ln_beta = nullptr;   // [H] fp32
    float ln_eps = 0.0f;
    bool ln_set = false;
    uint16_t* Xn = nullptr;  // [xn_rows][H] normalised block input
    int64_t xn_rows = 0;

    // backward pass
    float* zeros = nullptr;        // [max(H, F)] fp32 zeros: the "no bias" of dX
    float* colsum = nullptr;       // partial column sums for the bias gradients
    int64_t colsum_floats = 0;
    uint16_t* dgu = nullptr;       // gated backward: dG and dU, [rows][2F] bf16
    int64_t dgu_elems = 0;

    // split reduction of the last tiles on CTA pairs (absent with TPMLP_FLAG_FIXED_ORDER)
    float* sk_partial = nullptr;  // [num_sms / 2 pairs][2 units][2 CTAs][128 x 256] fp32 partials
    uint32_t* sk_count = nullptr; // [num_sms split tiles][2 CTAs][epilogue warps] arrivals
    uint32_t sk_epoch = 0;

    tpmlp::DeviceRates rates{};  // the planners' rates (device_rates, or tpmlp_set_device_rates)
    // row group of the tall units' sweep, for the last (512-row blocks, column blocks, pairs)
    int tall_group = 8, tall_group_m = -1, tall_group_n = -1, tall_group_pairs = -1;

    int* status = nullptr;  // device status word
    int64_t launches = 0;
    std::string last_error;
};

// Tile rasterisation: consecutive tiles walk down this many row blocks before moving to the
// next column block, so the CTAs that run at the same time share operand tiles in L2.
#ifndef TPMLP_GROUP_M1
#define TPMLP_GROUP_M1 16
#endif
// Split the reduction of the last tiles across all CTA pairs when the last wave of whole tiles
// would keep at most this percentage of the pairs busy.
#ifndef TPMLP_SPLIT_TAIL_PCT
#define TPMLP_SPLIT_TAIL_PCT 85
#endif
#ifndef TPMLP_GROUP_M2
#define TPMLP_GROUP_M2 8
#endif
// Operand-ring depth for 256-wide output tiles (48 KB per stage).
#ifndef TPMLP_STAGES_256
#define TPMLP_STAGES_256 4
#endif
// CTA-pair kernel: stages of 32 KB per CTA, and fp32 accumulators of 256 columns each.
#ifndef TPMLP_PAIR_STAGES
#define TPMLP_PAIR_STAGES 6
#endif
#ifndef TPMLP_PAIR_ACC
#define TPMLP_PAIR_ACC 2
#endif

namespace {

constexpr int kHostChunksMax = TPMLP_HOST_CHUNKS_MAX;  // row chunks of tpmlp_forward_host's pipeline

using tpmlp::GemmArgs;
using tpmlp::Mode;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

int fail_cuda(tpmlp_ctx* c, cudaError_t e, const char* what) {
    if (c) c->last_error = std::string(what) + ": " + cudaGetErrorString(e);
    return e == cudaErrorMemoryAllocation ? TPMLP_ERR_OOM : TPMLP_ERR_CUDA;
}

#define TPMLP_CUDA(ctx, call)                                   \
    do {                                                        \
        cudaError_t e_ = (call);                                \
        if (e_ != cudaSuccess) return fail_cuda(ctx, e_, #call); \
    } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int get_encoder(tpmlp_ctx* c) {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                        cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess && fn)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else if (g_encode_err == cudaSuccess)
            g_encode_err = cudaErrorSymbolNotFound;
    });
    if (!g_encode) return fail_cuda(c, g_encode_err, "cuTensorMapEncodeTiled entry point");
    return TPMLP_OK;
}

// bf16 tensor map with the 128-byte swizzle; dims/strides innermost first, strides in bytes
// for dims 1..rank-1. Out-of-range boxes are zero filled.
int encode_map(tpmlp_ctx* c, CUtensorMap* map, const void* ptr, int rank, const uint64_t* dims,
               const uint64_t* strides, const uint32_t* box) {
    int rc = get_encoder(c);
    if (rc) return rc;
    cuuint64_t d[3], s[2];
    cuuint32_t b[3], e[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i) s[i] = strides[i];
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), d, s,
                          b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        c->last_error = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(int(r));
        return TPMLP_ERR_CUDA;
    }
    return TPMLP_OK;
}

int pick_bn(int64_t width) {
    if (width % 256 == 0) return 256;
    if (width % 128 == 0) return 128;
    return 64;
}

// Opt a kernel into its dynamic shared memory once per device (bit d of `done`).
template <typename Kernel>
int ensure_smem_attr(tpmlp_ctx* c, Kernel kern, uint32_t smem, std::atomic<uint64_t>& done) {
    const uint64_t bit = uint64_t(1) << (c->device & 63);
    if (done.load(std::memory_order_acquire) & bit) return TPMLP_OK;
    TPMLP_CUDA(c, cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    done.fetch_or(bit, std::memory_order_acq_rel);
    return TPMLP_OK;
}

// Launch a GEMM kernel with programmatic stream serialisation: its CTAs may be scheduled while
// the kernel before it in the stream finishes, run their set-up (barriers, tensor memory,
// descriptor prefetch), and wait in griddep_wait until that kernel's results are visible.
// b2: the B map of shards [args.k2, args.k) of a second-GEMM reduction (unused otherwise).
template <typename Kernel>
cudaError_t launch_overlapped(Kernel kern, int grid, uint32_t smem, cudaStream_t s,
                              const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2,
                              const GemmArgs& args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(tpmlp::kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a, b, b2, args);
}

template <int BN, int STAGES, Mode MODE, bool F32, bool MN = false>
int launch_gemm(tpmlp_ctx* c, const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& args,
                cudaStream_t s, const CUtensorMap* b2 = nullptr) {
    auto kern = tpmlp::tpmlp_gemm_kernel<BN, STAGES, MODE, F32, MN>;
    constexpr uint32_t smem = tpmlp::GemmSmem<BN, STAGES>::kTotal;
    static std::atomic<uint64_t> attr_done{0};
    if (int rc = ensure_smem_attr(c, kern, smem, attr_done)) return rc;
    const int grid = std::min(args.num_tiles, c->num_sms);
    TPMLP_CUDA(c, launch_overlapped(kern, grid, smem, s, a, b, b2 ? *b2 : b, args));
    ++c->launches;
    return TPMLP_OK;
}

// Stage depth per tile width: 192 KB of operand ring in every case.
template <Mode MODE, bool F32>
int dispatch_gemm(tpmlp_ctx* c, int bn, const CUtensorMap& a, const CUtensorMap& b,
                  const GemmArgs& args, cudaStream_t s, const CUtensorMap* b2 = nullptr) {
    switch (bn) {
        case 256: return launch_gemm<256, TPMLP_STAGES_256, MODE, F32>(c, a, b, args, s, b2);
        case 128: return launch_gemm<128, 6, MODE, F32>(c, a, b, args, s, b2);
        default:
            // the gated layer's tiles hold 2 x 64 columns at least
            if constexpr (tpmlp::is_gated(MODE)) return TPMLP_ERR_UNSUPPORTED_SHAPE;
            else return launch_gemm<64, 8, MODE, F32>(c, a, b, args, s, b2);
    }
}

// Largest number of CTA pairs of this kernel that can be resident at once.
template <typename Kernel>
int max_resident_pairs(tpmlp_ctx* c, Kernel kern, uint32_t smem) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (c->num_sms / 2), 1, 1);
    cfg.blockDim = dim3(tpmlp::kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();  // clear; fall back to one pair per two SMs
        n = c->num_sms / 2;
    }
    return n;
}

// The split plan of one pair-kernel launch (GemmArgs::sk_*, tpmlp_plan.h). Measured against
// whole tiles:
//  - Launches of one to two waves, split entirely: the GPT-2 second GEMM (96 tiles, 55 MB of
//    operands, 48 blocks) 10 % faster. The 7b second GEMM on 2048-row chunks (128 tiles,
//    201 MB) and the GPT-2 first GEMM on 2048-row chunks (96 tiles, 12 blocks) were slower,
//    hence the L2 and depth limits.
//  - Longer launches: splitting a whole wave plus the tail (132 of the 7b second GEMM's 512
//    tiles) cost 9 %, because the pairs' staggered shares lose the wave's shared operands in
//    L2. Only the last R tiles are split, and only where the model (R / P of a round plus
//    one DRAM read of the tail's operands, under half a round) favours it: the GPT-3 second
//    GEMM (R = 8, 768 blocks) 4.7 % faster; the GPT-3 first GEMM (R = 32, 192 blocks, at 70 %
//    of a round by the model) 1.3 % slower, hence the half.
// The rule's rates are the context's (device_rates at create, or tpmlp_set_device_rates).
tpmlp::SplitRule split_rule_of(const tpmlp_ctx* c, int pairs) {
    tpmlp::SplitRule r = tpmlp::split_rule(c->rates, pairs);
    r.tail_pct = TPMLP_SPLIT_TAIL_PCT;
    return r;
}

// The split's flags carry an epoch chosen here, per launch. A launch recorded into a CUDA graph
// would replay with the same epoch and could read partial sums before they are written, so
// launches enqueued under stream capture never split.
bool capturing(cudaStream_t s) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) != cudaSuccess) {
        cudaGetLastError();
        return true;  // unknown: take the safe path
    }
    return st != cudaStreamCaptureStatusNone;
}

// Returns the number of pairs to launch: min(T, resident), or the plan's count when a launch
// of fewer tiles than pairs spreads each tile over several pairs.
int plan_split(tpmlp_ctx* c, GemmArgs& a, int resident, cudaStream_t s) {
    a.sk_first = a.num_tiles;
    a.sk_iters = 0;
    const int pairs = std::min(a.num_tiles, resident);
    if (!c->sk_partial || resident > c->num_sms / 2 || capturing(s)) return pairs;
    const tpmlp::SplitLaunch L{a.num_tiles, resident, a.kb_tile,       a.m_blocks,
                               a.n_blocks,  a.group_m, tpmlp::kPairBM, tpmlp::kPairBN};
    const tpmlp::SplitPlan p = tpmlp::plan_split_tiles(L, split_rule_of(c, c->num_sms / 2));
    // the counters hold num_sms split tiles (the plan never splits more than 2 * pairs)
    if (p.sk_first == a.num_tiles || a.num_tiles - p.sk_first > c->num_sms) return pairs;
    if (p.pairs > resident) return pairs;
    a.sk_first = p.sk_first;
    a.sk_iters = p.sk_iters;
    a.sk_partial = c->sk_partial;
    a.sk_count = c->sk_count;
    if (++c->sk_epoch == 0) c->sk_epoch = 1;  // counters start at 0 (epoch 0): never reuse it
    a.sk_epoch = c->sk_epoch;
    return p.pairs > 0 ? p.pairs : pairs;
}

template <int STAGES, int NUM_ACC, Mode MODE, bool F32, bool MN = false>
int launch_pair(tpmlp_ctx* c, const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& args,
                cudaStream_t s, const CUtensorMap* b2 = nullptr) {
    auto kern = tpmlp::tpmlp_gemm_pair_kernel<STAGES, NUM_ACC, MODE, F32, MN>;
    constexpr uint32_t smem = tpmlp::PairSmem<STAGES, NUM_ACC>::kTotal;
    static_assert(smem <= 232448, "shared memory per CTA");
    static std::atomic<uint64_t> attr_done{0};
    if (int rc = ensure_smem_attr(c, kern, smem, attr_done)) return rc;
    static std::atomic<int> resident_on[64];  // per device, looked up on first use (0: not yet)
    std::atomic<int>& slot = resident_on[c->device & 63];
    int resident = slot.load(std::memory_order_relaxed);
    if (resident <= 0) {
        resident = max_resident_pairs(c, kern, smem);
        slot.store(resident, std::memory_order_relaxed);
    }
    GemmArgs run = args;
    const int pairs = plan_split(c, run, resident, s);
    TPMLP_CUDA(c, launch_overlapped(kern, 2 * pairs, smem, s, a, b, b2 ? *b2 : b, run));
    ++c->launches;
    return TPMLP_OK;
}

// The packed second-layer weight of a context whose second GEMM runs on CTA pairs is stored
// in 16 KB blocks (transpose_blocked_bf16_kernel): one TMA box of the pair kernel (128 rows x
// 64 reduction columns) is then one contiguous block instead of 128 pieces of 128 bytes spread
// over 128 rows. Interleaved A/B against the row-major [k][H][f] layout, bit-identical output:
// second GEMM 588.8 -> 580.7 us at 7b, 2869 -> 2808 us at GPT-3, 1246 -> 1226 us on the
// sweep's 16384 tokens; GPT-2 unchanged.
bool w2_blocked(const tpmlp_ctx* c) { return c->pair2; }

// The second GEMM on CTA pairs. Reductions at least TPMLP_TALL_MIN_KB blocks deep run their
// whole waves of 512 x 256 tall units with the TALL kernel (4 stages of 48 KB: two A halves and
// one shared B tile), and the rest of the output as ordinary tiles in the same launch, split
// over all pairs when the tail rule says so (tpmlp_plan.h, plan_tall_units).
#ifndef TPMLP_TALL_MIN_KB
#define TPMLP_TALL_MIN_KB 128
#endif
#ifndef TPMLP_TALL_STAGES
#define TPMLP_TALL_STAGES 4
#endif
template <Mode MODE, bool F32>
int launch_gemm2_pair(tpmlp_ctx* c, const CUtensorMap& a_map, const CUtensorMap& b_map,
                      const GemmArgs& args, cudaStream_t s, const CUtensorMap* b2 = nullptr) {
    if (args.kb_tile >= TPMLP_TALL_MIN_KB) {
        auto kern = tpmlp::tpmlp_gemm_pair_kernel<TPMLP_TALL_STAGES, 2, MODE, F32, false, true>;
        constexpr uint32_t smem = tpmlp::PairSmem<TPMLP_TALL_STAGES, 2, true>::kTotal;
        static_assert(smem <= 232448, "shared memory per CTA");
        static std::atomic<uint64_t> attr_done{0};
        if (int rc = ensure_smem_attr(c, kern, smem, attr_done)) return rc;
        static std::atomic<int> resident_on[64];
        std::atomic<int>& slot = resident_on[c->device & 63];
        int resident = slot.load(std::memory_order_relaxed);
        if (resident <= 0) {
            resident = max_resident_pairs(c, kern, smem);
            slot.store(resident, std::memory_order_relaxed);
        }
        // the row group of the units' sweep: the one whose rounds read the least from DRAM
        const int tall_m = args.M / (2 * tpmlp::kPairBM);
        if (tall_m != c->tall_group_m || args.n_blocks != c->tall_group_n ||
            resident != c->tall_group_pairs) {
            c->tall_group = tpmlp::pick_tall_group(tall_m, args.n_blocks, resident);
            c->tall_group_m = tall_m;
            c->tall_group_n = args.n_blocks;
            c->tall_group_pairs = resident;
        }
        const int group = c->tall_group;
        const tpmlp::TallPlan tall = tpmlp::plan_tall_units(args.M, args.n_blocks, group, resident);
        if (tall.tall_units > 0) {
            GemmArgs run = args;
            run.group_m = group;
            // every second round sweeps the reduction backwards, except in the fixed order
            run.tall_serpentine = (c->flags & TPMLP_FLAG_FIXED_ORDER) ? 0 : 1;
            run.tall_units = tall.tall_units;
            run.tall_m_blocks = tall.tall_m_blocks;
            run.tall_rest = tall.tall_rest;
            run.num_tiles = tall.tiles;
            run.sk_first = tall.tiles;  // the remaining tiles whole ...
            run.sk_iters = 0;
            // ... except their last, partial wave, spread over all pairs when that pays
            const int whole = tall.tail_first, rem = tall.tiles - whole;
            if (c->sk_partial && resident <= c->num_sms / 2 && !capturing(s) && rem > 0 &&
                rem <= c->num_sms &&
                tpmlp::tail_split_pays(rem, args.kb_tile, resident, tall.rows, tall.cols,
                                       tpmlp::kPairBM, tpmlp::kPairBN,
                                       split_rule_of(c, c->num_sms / 2))) {
                run.sk_first = whole;
                run.sk_iters = rem * args.kb_tile;
                run.sk_partial = c->sk_partial;
                run.sk_count = c->sk_count;
                if (++c->sk_epoch == 0) c->sk_epoch = 1;
                run.sk_epoch = c->sk_epoch;
            }
            TPMLP_CUDA(c, launch_overlapped(kern, 2 * resident, smem, s, a_map, b_map,
                                            b2 ? *b2 : b_map, run));
            ++c->launches;
            return TPMLP_OK;
        }
    }
    return launch_pair<TPMLP_PAIR_STAGES, TPMLP_PAIR_ACC, MODE, F32>(c, a_map, b_map, args, s, b2);
}

GemmArgs base_args(const tpmlp_ctx* c, int64_t M, int ldo, int bm, int bn, int group_m) {
    GemmArgs a{};
    a.M = static_cast<int>(M);
    a.ldo = ldo;
    a.f = static_cast<int>(c->f);
    a.k = c->k;
    a.m_blocks = static_cast<int>((M + bm - 1) / bm);
    a.n_blocks = ldo / bn;
    a.num_tiles = a.m_blocks * a.n_blocks;
    a.group_m = group_m;
    a.status = c->status;
    a.ldo2 = ldo;
    a.half = 0;
    a.k2 = c->k;
    a.sk_first = a.num_tiles;  // no split (set per launch by plan_split)
    return a;
}

constexpr int kKindBlock = 0, kKindColumn = 1, kKindRow = 2;

#ifdef TPMLP_TEST_HOOKS
// Test builds only: a device index that the current-device query reports instead of the real
// one (-1: the real one), so that host tests drive the device check without a GPU.
std::atomic<int> g_test_current_device{-1};
#endif

cudaError_t current_device(int* dev) {
#ifdef TPMLP_TEST_HOOKS
    const int fake = g_test_current_device.load();
    if (fake >= 0) {
        *dev = fake;
        return cudaSuccess;
    }
#endif
    return cudaGetDevice(dev);
}

// The context's device must be current on the calling thread: the context's buffers, tensor
// maps and kernel attributes belong to that device, and a launch would otherwise run on
// another GPU with them. Every entry point that enqueues work or touches the context's device
// memory checks this first.
int check_device(tpmlp_ctx* c) {
    int cur = -1;
    const cudaError_t e = current_device(&cur);
    if (e != cudaSuccess) return fail_cuda(c, e, "cudaGetDevice");
    if (cur != c->device) {
        c->last_error = "the context belongs to device " + std::to_string(c->device) + " but device " +
                        std::to_string(cur) + " is current (call cudaSetDevice first)";
        return TPMLP_ERR_INVALID_ARG;
    }
    return TPMLP_OK;
}

// An MLP-block context on the current device whose weights are packed.
int check_ctx(tpmlp_ctx* c) {
    if (!c || c->kind != kKindBlock) return TPMLP_ERR_INVALID_ARG;
    if (int rc = check_device(c)) return rc;
    if (!c->packed) return TPMLP_ERR_NOT_PACKED;
    return TPMLP_OK;
}

// Tensor map of a row-major bf16 [rows][cols] activation, box 64 x 128, cached per pointer
// and row count.
int activation_map(tpmlp_ctx* c, const void* ptr, int64_t rows, int64_t cols,
                   const void*& cached_ptr, int64_t& cached_rows, CUtensorMap& map) {
    if (ptr == cached_ptr && rows == cached_rows) return TPMLP_OK;
    const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)};
    const uint64_t strides[1] = {static_cast<uint64_t>(cols) * 2};
    const uint32_t box[2] = {tpmlp::kBK, tpmlp::kBM};
    cached_ptr = nullptr;
    int rc = encode_map(c, &map, ptr, 2, dims, strides, box);
    if (rc) return rc;
    cached_ptr = ptr;
    cached_rows = rows;
    return TPMLP_OK;
}

int run_gemm1(tpmlp_ctx* c, const void* X, int64_t M, void* Y, cudaStream_t s,
              bool linear = false, void* A_save = nullptr) {
    int rc = activation_map(c, X, M, c->H, c->x_map_ptr, c->x_map_rows, c->tmX);
    if (rc) return rc;
    const CUtensorMap& tmX = c->tmX;
    const bool pair = c->pair1;
    const int tile_rows_b = pair ? tpmlp::kPairBN : c->bn1;  // B rows (output columns) per tile
    GemmArgs a = base_args(c, M, static_cast<int>(c->F), pair ? tpmlp::kPairBM : tpmlp::kBM,
                           tile_rows_b, TPMLP_GROUP_M1);
    a.kb_tile = static_cast<int>(c->H / tpmlp::kBK);
    a.kb_shard = a.kb_tile;
    a.bias = c->b1;
    a.out = Y;
    if (c->gated) {
        // tiles walk the 2F packed rows; each yields half as many output columns
        a.f = static_cast<int>(2 * c->f);
        a.n_blocks = static_cast<int>(2 * c->F / tile_rows_b);
        a.num_tiles = a.m_blocks * a.n_blocks;
        if (A_save) {
            // training forward: also keep G and U, [M][2F] (U from column F on)
            a.out2 = A_save;
            a.ldo2 = static_cast<int>(2 * c->F);
            a.half = static_cast<int>(c->F);
            if (pair)
                return launch_pair<TPMLP_PAIR_STAGES, TPMLP_PAIR_ACC, Mode::kGemm1GatedTrain, false>(
                    c, tmX, c->tmW1_pair, a, s);
            return dispatch_gemm<Mode::kGemm1GatedTrain, false>(c, c->bn1, tmX, c->tmW1, a, s);
        }
        if (pair)
            return launch_pair<TPMLP_PAIR_STAGES, TPMLP_PAIR_ACC, Mode::kGemm1Gated, false>(
                c, tmX, c->tmW1_pair, a, s);
        return dispatch_gemm<Mode::kGemm1Gated, false>(c, c->bn1, tmX, c->tmW1, a, s);
    }
    if (A_save) {
        // training forward: also keep the pre-activation for the backward pass
        a.out2 = A_save;
        if (pair)
            return launch_pair<TPMLP_PAIR_STAGES, TPMLP_PAIR_ACC, Mode::kGemm1Train, false>(
                c, tmX, c->tmW1_pair, a, s);
        return dispatch_gemm<Mode::kGemm1Train, false>(c, c->bn1, tmX, c->tmW1, a, s);
    }
    if (linear) {
        // column-parallel linear layer: bias only, output bf16 or fp32
        if (c->flags & TPMLP_FLAG_Z_FP32) {
            if (pair)
                return launch_pair<TPMLP_PAIR_STAGES, TPMLP_PAIR_ACC, Mode::kGemm1Linear, true>(
                    c, tmX, c->tmW1_pair, a, s);
            return dispatch_gemm<Mode::kGemm1Linear, true>(c, c->bn1, tmX, c->tmW1, a, s);
        }
        if (pair)
            return launch_pair<TPMLP_PAIR_STAGES, TPMLP_PAIR_ACC, Mode::kGemm1Linear, false>(
                c, tmX, c->tmW1_pair, a, s);
        return dispatch_gemm<Mode::kGemm1Linear, false>(c, c->bn1, tmX, c->tmW1, a, s);
    }
    if (pair)
        return launch_pair<TPMLP_PAIR_STAGES, TPMLP_PAIR_ACC, Mode::kGemm1, false>(c, tmX,
                                                                                   c->tmW1_pair, a, s);
    return dispatch_gemm<Mode::kGemm1, false>(c, c->bn1, tmX, c->tmW1, a, s);
}

int run_gemm2(tpmlp_ctx* c, const void* Y, int64_t M, void* Z, cudaStream_t s,
              const void* residual = nullptr) {
    int rc = activation_map(c, Y, M, c->F, c->y_map_ptr, c->y_map_rows, c->tmY);
    if (rc) return rc;
    const CUtensorMap& tmY = c->tmY;
    const bool pair = c->pair2;
    GemmArgs a = base_args(c, M, static_cast<int>(c->H), pair ? tpmlp::kPairBM : tpmlp::kBM,
                           pair ? tpmlp::kPairBN : c->bn2, TPMLP_GROUP_M2);
    a.kb_shard = static_cast<int>(c->f / tpmlp::kBK);
    a.kb_tile = a.kb_shard * c->k;
    a.bias = c->b2;
    a.out = Z;
    a.residual = residual;
    a.b_blocked = w2_blocked(c) ? 1 : 0;
    if (residual) {
        if (pair) {
            if (c->flags & TPMLP_FLAG_Z_FP32)
                return launch_gemm2_pair<Mode::kGemm2Residual, true>(c, tmY, c->tmW2_pair, a, s);
            return launch_gemm2_pair<Mode::kGemm2Residual, false>(c, tmY, c->tmW2_pair, a, s);
        }
        if (c->flags & TPMLP_FLAG_Z_FP32)
            return dispatch_gemm<Mode::kGemm2Residual, true>(c, c->bn2, tmY, c->tmW2, a, s);
        return dispatch_gemm<Mode::kGemm2Residual, false>(c, c->bn2, tmY, c->tmW2, a, s);
    }
    if (pair) {
        if (c->flags & TPMLP_FLAG_Z_FP32)
            return launch_gemm2_pair<Mode::kGemm2, true>(c, tmY, c->tmW2_pair, a, s);
        return launch_gemm2_pair<Mode::kGemm2, false>(c, tmY, c->tmW2_pair, a, s);
    }
    if (c->flags & TPMLP_FLAG_Z_FP32)
        return dispatch_gemm<Mode::kGemm2, true>(c, c->bn2, tmY, c->tmW2, a, s);
    return dispatch_gemm<Mode::kGemm2, false>(c, c->bn2, tmY, c->tmW2, a, s);
}

int ensure_y(tpmlp_ctx* c, int64_t rows) {
    if (rows <= c->y_rows) return TPMLP_OK;
    const int64_t want = ((rows + tpmlp::kBM - 1) / tpmlp::kBM) * tpmlp::kBM;
    TPMLP_CUDA(c, cudaDeviceSynchronize());  // the old buffer may still be in use
    if (c->Y) cudaFree(c->Y);
    c->Y = nullptr;
    c->y_rows = 0;
    TPMLP_CUDA(c, cudaMalloc(&c->Y, static_cast<size_t>(want) * c->F * 2));
    c->y_rows = want;
    return TPMLP_OK;
}

int check_tokens(int64_t B, int64_t S) {
    if (B < 0 || S < 0) return TPMLP_ERR_INVALID_ARG;
    if (S > 0 && B > (int64_t(1) << 31) / S) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    return TPMLP_OK;
}

int z_elem_bytes(const tpmlp_ctx* c) { return (c->flags & TPMLP_FLAG_Z_FP32) ? 4 : 2; }

// Row chunks of tpmlp_forward_host for M tokens (tpmlp_plan.h), timed with the context's rates.
int plan_host_chunks(const tpmlp_ctx* c, int64_t M, int64_t* rows) {
    tpmlp::ChunkModel m{};
    const int64_t pairs = c->num_sms / 2;
    const int64_t F1 = c->gated ? 2 * c->F : c->F;  // first GEMM's output columns (packed)
    const int64_t K[2] = {c->H, c->F}, N[2] = {F1, c->H};
    const bool pair[2] = {c->pair1, c->pair2};
    const int64_t bn[2] = {c->bn1, c->bn2};
    for (int i = 0; i < 2; ++i) {
        tpmlp::ChunkGemm& g = m.g[i];
        g.tile_rows = pair[i] ? tpmlp::kPairBM : tpmlp::kBM;
        const int64_t w = pair[i] ? tpmlp::kPairBN : bn[i];
        g.col_tiles = N[i] / w;
        g.slots = pair[i] ? pairs : c->num_sms;
        g.tile_s = 2.0 * g.tile_rows * w * K[i] / (c->rates.gemm_flops / g.slots);
        g.launch_s = tpmlp::kChunkLaunchS;
    }
    m.x_row_bytes = 2.0 * c->H;
    m.z_row_bytes = static_cast<double>(c->H) * z_elem_bytes(c);
    m.copy_Bps = c->rates.copy_Bps;
    return tpmlp::plan_chunks(m, M, kHostChunksMax, 64, rows);
}

// W2 [F][H] = k blocks [f][H] -> W2p [k][H][f] (or in 16 KB blocks); b2 -> fp32.
int pack_second_layer(tpmlp_ctx* c, const void* W2, const void* b2, cudaStream_t s) {
    const int T = tpmlp::kTransposeTile;
    dim3 grid(static_cast<unsigned>(c->H / T), static_cast<unsigned>(c->f / T),
              static_cast<unsigned>(c->k));
    if (w2_blocked(c))
        tpmlp::transpose_blocked_bf16_kernel<<<grid, dim3(64, 4), 0, s>>>(
            static_cast<const uint16_t*>(W2), c->W2p, static_cast<int>(c->f), static_cast<int>(c->H));
    else
        tpmlp::transpose_bf16_kernel<<<grid, dim3(64, 4), 0, s>>>(
            static_cast<const uint16_t*>(W2), c->W2p, static_cast<int>(c->f), static_cast<int>(c->H),
            static_cast<long long>(c->f) * c->H, static_cast<long long>(c->f) * c->H);
    TPMLP_CUDA(c, cudaGetLastError());
    tpmlp::bf16_to_f32_kernel<<<static_cast<unsigned>((c->H + 255) / 256), 256, 0, s>>>(
        static_cast<const uint16_t*>(b2), c->b2, c->H);
    TPMLP_CUDA(c, cudaGetLastError());
    c->launches += 2;
    return TPMLP_OK;
}

// Tensor maps of the packed shards: box 64 (reduction) x rows x 1 shard, for the single-SM
// kernel (rows = its tile width) and for the CTA-pair kernel (rows = 128 per CTA).
int encode_weight_maps(tpmlp_ctx* c) {
    if (c->W1p) {
        const int64_t rows1 = c->gated ? 2 * c->f : c->f;  // packed rows per shard
        const uint64_t dims[3] = {static_cast<uint64_t>(c->H), static_cast<uint64_t>(rows1),
                                  static_cast<uint64_t>(c->k)};
        const uint64_t strides[2] = {static_cast<uint64_t>(c->H) * 2,
                                     static_cast<uint64_t>(rows1) * c->H * 2};
        const uint32_t box[3] = {tpmlp::kBK, static_cast<uint32_t>(c->bn1), 1};
        int rc = encode_map(c, &c->tmW1, c->W1p, 3, dims, strides, box);
        if (rc) return rc;
        const uint32_t box_pair[3] = {tpmlp::kBK, 128, 1};
        rc = encode_map(c, &c->tmW1_pair, c->W1p, 3, dims, strides, box_pair);
        if (rc) return rc;
    }
    if (c->W2p) {
        const uint64_t dims[3] = {static_cast<uint64_t>(c->f), static_cast<uint64_t>(c->H),
                                  static_cast<uint64_t>(c->k)};
        const uint64_t strides[2] = {static_cast<uint64_t>(c->f) * 2,
                                     static_cast<uint64_t>(c->f) * c->H * 2};
        const uint32_t box[3] = {tpmlp::kBK, static_cast<uint32_t>(c->bn2), 1};
        int rc = encode_map(c, &c->tmW2, c->W2p, 3, dims, strides, box);
        if (rc) return rc;
        if (w2_blocked(c)) {
            // 128-byte rows, 128 of them per box: one 16 KB block
            const uint64_t bdims[2] = {static_cast<uint64_t>(tpmlp::kBK),
                                       static_cast<uint64_t>(c->k) * c->H * (c->f / tpmlp::kBK)};
            const uint64_t bstrides[1] = {static_cast<uint64_t>(tpmlp::kBK) * 2};
            const uint32_t bbox[2] = {tpmlp::kBK, 128};
            rc = encode_map(c, &c->tmW2_pair, c->W2p, 2, bdims, bstrides, bbox);
        } else {
            const uint32_t box_pair[3] = {tpmlp::kBK, 128, 1};
            rc = encode_map(c, &c->tmW2_pair, c->W2p, 3, dims, strides, box_pair);
        }
        if (rc) return rc;
    }
    return TPMLP_OK;
}

int ensure_xn(tpmlp_ctx* c, int64_t rows) {
    if (rows <= c->xn_rows) return TPMLP_OK;
    const int64_t want = ((rows + tpmlp::kBM - 1) / tpmlp::kBM) * tpmlp::kBM;
    TPMLP_CUDA(c, cudaDeviceSynchronize());  // the old buffer may still be in use
    if (c->Xn) cudaFree(c->Xn);
    c->Xn = nullptr;
    c->xn_rows = 0;
    TPMLP_CUDA(c, cudaMalloc(&c->Xn, static_cast<size_t>(want) * c->H * 2));
    c->xn_rows = want;
    return TPMLP_OK;
}

template <int THREADS, int NC>
void launch_layernorm(const tpmlp_ctx* c, const void* X, int64_t M, void* Xn, cudaStream_t s) {
    tpmlp::layernorm_kernel<THREADS, NC><<<static_cast<unsigned>(M), THREADS, 0, s>>>(
        static_cast<const uint16_t*>(X), c->ln_gamma, c->ln_beta, c->ln_eps,
        static_cast<uint16_t*>(Xn), static_cast<int>(c->H));
}

// CTA size by row length (measured: 64 / 128 / 256 threads best for H <= 4096 / 8192 / more);
// NC = 16-byte chunks per thread, rounded up to an instantiated count.
int run_layernorm(tpmlp_ctx* c, const void* X, int64_t M, void* Xn, cudaStream_t s) {
    const int64_t chunks = c->H / 8;
    if (c->H <= 4096) {
        switch ((chunks + 63) / 64) {
            case 1: launch_layernorm<64, 1>(c, X, M, Xn, s); break;
            case 2: launch_layernorm<64, 2>(c, X, M, Xn, s); break;
            case 3: launch_layernorm<64, 3>(c, X, M, Xn, s); break;
            case 4: launch_layernorm<64, 4>(c, X, M, Xn, s); break;
            case 5: case 6: launch_layernorm<64, 6>(c, X, M, Xn, s); break;
            default: launch_layernorm<64, 8>(c, X, M, Xn, s); break;
        }
    } else if (c->H <= 8192) {
        switch ((chunks + 127) / 128) {
            case 5: case 6: launch_layernorm<128, 6>(c, X, M, Xn, s); break;
            default: launch_layernorm<128, 8>(c, X, M, Xn, s); break;
        }
    } else if (c->H <= tpmlp::kNormMaxH) {
        switch ((chunks + 255) / 256) {
            case 5: case 6: launch_layernorm<256, 6>(c, X, M, Xn, s); break;
            default: launch_layernorm<256, 8>(c, X, M, Xn, s); break;
        }
    } else {
        return TPMLP_ERR_UNSUPPORTED_SHAPE;
    }
    TPMLP_CUDA(c, cudaGetLastError());
    ++c->launches;
    return TPMLP_OK;
}

// The copy streams and events of the host-buffer entry points, created on first use. After a
// failure the next call creates only what is still missing; tpmlp_destroy releases them all.
int ensure_copy_streams(tpmlp_ctx* c) {
    if (c->s_in && c->s_out) return TPMLP_OK;
    auto event = [c](cudaEvent_t& e) -> int {
        if (!e) TPMLP_CUDA(c, cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
        return TPMLP_OK;
    };
    int rc;
    for (cudaEvent_t& e : c->host_ev)
        if ((rc = event(e))) return rc;
    for (int i = 0; i < kHostChunksMax; ++i)
        if ((rc = event(c->in_ev[i])) || (rc = event(c->out_ev[i]))) return rc;
    for (int i = 0; i < 2; ++i)
        if ((rc = event(c->a_in[i])) || (rc = event(c->a_xfree[i])) ||
            (rc = event(c->a_zready[i])) || (rc = event(c->a_zfree[i])))
            return rc;
    if (!c->s_in) TPMLP_CUDA(c, cudaStreamCreateWithFlags(&c->s_in, cudaStreamNonBlocking));
    if (!c->s_out) TPMLP_CUDA(c, cudaStreamCreateWithFlags(&c->s_out, cudaStreamNonBlocking));
    return TPMLP_OK;
}

// The host-buffer entry points queue work on the context's own copy streams, which a CUDA
// graph capture of `s` cannot take in; they refuse to run under capture.
int refuse_capture(tpmlp_ctx* c, cudaStream_t s) {
    if (!capturing(s)) return TPMLP_OK;
    c->last_error = "host-buffer entry points cannot run under stream capture";
    return TPMLP_ERR_INVALID_ARG;
}

// The host-buffer pipeline of tpmlp_forward_host (layer = false) and
// tpmlp_block_forward_host (layer = true: LayerNorm in front, the residual added by the second
// GEMM's epilogue). The planned row chunks of X are copied into a device staging buffer on one
// copy stream, each chunk's kernels run on `s` once its rows have arrived, and each chunk of Z
// is copied out on a second copy stream as soon as its second GEMM is done.
int run_host_pipeline(tpmlp_ctx* c, const void* X_host, int64_t B, int64_t S, void* Z_host,
                      cudaStream_t s, bool layer) {
    int rc = check_ctx(c);
    if (rc) return rc;
    if (layer && !c->ln_set) {
        c->last_error = "LayerNorm parameters not set (tpmlp_set_layernorm)";
        return TPMLP_ERR_NOT_PACKED;
    }
    if ((rc = check_tokens(B, S))) return rc;
    const int64_t M = B * S;
    if (M == 0) return TPMLP_OK;
    if ((rc = refuse_capture(c, s))) return rc;
    if (!X_host || !Z_host) return TPMLP_ERR_INVALID_ARG;
    if (M > (int64_t(1) << 31) - 1) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    if (M > c->stage_rows) {
        TPMLP_CUDA(c, cudaDeviceSynchronize());
        if (c->Xs) cudaFree(c->Xs);
        if (c->Zs) cudaFree(c->Zs);
        c->Xs = c->Zs = nullptr;
        c->stage_rows = 0;
        TPMLP_CUDA(c, cudaMalloc(&c->Xs, static_cast<size_t>(M) * c->H * 2));
        TPMLP_CUDA(c, cudaMalloc(&c->Zs, static_cast<size_t>(M) * c->H * z_elem_bytes(c)));
        c->stage_rows = M;
    }
    if ((rc = ensure_y(c, M))) return rc;
    if (layer && (rc = ensure_xn(c, M))) return rc;
    if ((rc = ensure_copy_streams(c))) return rc;
    if (M != c->plan_M) {
        c->plan_n = plan_host_chunks(c, M, c->plan_rows);
        c->plan_M = M;
    }
    const size_t xrow = static_cast<size_t>(c->H) * 2, zrow = static_cast<size_t>(c->H) * z_elem_bytes(c);
    // nothing may touch the staging buffers before earlier work on `s` is done
    TPMLP_CUDA(c, cudaEventRecord(c->host_ev[0], s));
    TPMLP_CUDA(c, cudaStreamWaitEvent(c->s_in, c->host_ev[0], 0));
    TPMLP_CUDA(c, cudaStreamWaitEvent(c->s_out, c->host_ev[0], 0));
    int64_t r0 = 0;
    for (int i = 0; i < c->plan_n; ++i) {
        const int64_t n = c->plan_rows[i];
        TPMLP_CUDA(c, cudaMemcpyAsync(static_cast<char*>(c->Xs) + r0 * xrow,
                                      static_cast<const char*>(X_host) + r0 * xrow, n * xrow,
                                      cudaMemcpyHostToDevice, c->s_in));
        TPMLP_CUDA(c, cudaEventRecord(c->in_ev[i], c->s_in));
        r0 += n;
    }
    r0 = 0;
    for (int i = 0; i < c->plan_n; ++i) {
        const int64_t n = c->plan_rows[i];
        TPMLP_CUDA(c, cudaStreamWaitEvent(s, c->in_ev[i], 0));
        const void* xi = static_cast<const char*>(c->Xs) + r0 * xrow;
        void* zi = static_cast<char*>(c->Zs) + r0 * zrow;
        if (layer) {
            if ((rc = run_layernorm(c, xi, n, c->Xn, s)) || (rc = run_gemm1(c, c->Xn, n, c->Y, s)) ||
                (rc = run_gemm2(c, c->Y, n, zi, s, xi)))
                return rc;
        } else if ((rc = run_gemm1(c, xi, n, c->Y, s)) || (rc = run_gemm2(c, c->Y, n, zi, s))) {
            return rc;
        }
        TPMLP_CUDA(c, cudaEventRecord(c->out_ev[i], s));
        TPMLP_CUDA(c, cudaStreamWaitEvent(c->s_out, c->out_ev[i], 0));
        TPMLP_CUDA(c, cudaMemcpyAsync(static_cast<char*>(Z_host) + r0 * zrow, zi, n * zrow,
                                      cudaMemcpyDeviceToHost, c->s_out));
        r0 += n;
    }
    TPMLP_CUDA(c, cudaEventRecord(c->host_ev[1], c->s_out));
    TPMLP_CUDA(c, cudaStreamWaitEvent(s, c->host_ev[1], 0));
    TPMLP_CUDA(c, cudaStreamSynchronize(s));
    return TPMLP_OK;
}

// tpmlp_forward_host_async (layer = false) and tpmlp_block_forward_host_async (layer = true):
// the whole call as one chunk in staging slot (calls made so far) mod 2. Its input copy on the
// context's input stream waits only until the kernels of the call before last have read the
// slot, and its output copy on the output stream only for this call's second GEMM, so that in
// a run of calls the copies of one call overlap the kernels of its neighbours. Nothing here
// waits on the host; tpmlp_host_wait does.
int run_host_async(tpmlp_ctx* c, const void* X_host, int64_t B, int64_t S, void* Z_host,
                   cudaStream_t s, bool layer) {
    int rc = check_ctx(c);
    if (rc) return rc;
    if (layer && !c->ln_set) {
        c->last_error = "LayerNorm parameters not set (tpmlp_set_layernorm)";
        return TPMLP_ERR_NOT_PACKED;
    }
    if ((rc = check_tokens(B, S))) return rc;
    const int64_t M = B * S;
    if (M == 0) return TPMLP_OK;
    if ((rc = refuse_capture(c, s))) return rc;
    if (!X_host || !Z_host) return TPMLP_ERR_INVALID_ARG;
    if (M > (int64_t(1) << 31) - 1) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    if ((rc = ensure_copy_streams(c))) return rc;
    const size_t xbytes = static_cast<size_t>(M) * c->H * 2;
    const size_t zbytes = static_cast<size_t>(M) * c->H * z_elem_bytes(c);
    if (M > c->async_rows) {
        TPMLP_CUDA(c, cudaDeviceSynchronize());  // earlier calls may still use the slots
        for (int i = 0; i < 2; ++i) {
            cudaFree(c->Xa[i]);
            cudaFree(c->Za[i]);
            c->Xa[i] = c->Za[i] = nullptr;
            c->a_used[i] = false;
        }
        c->async_rows = 0;
        for (int i = 0; i < 2; ++i) {
            TPMLP_CUDA(c, cudaMalloc(&c->Xa[i], xbytes));
            TPMLP_CUDA(c, cudaMalloc(&c->Za[i], zbytes));
        }
        c->async_rows = M;
    }
    if ((rc = ensure_y(c, M))) return rc;
    if (layer && (rc = ensure_xn(c, M))) return rc;
    const int slot = static_cast<int>(c->a_calls & 1u);
    void* const xs = c->Xa[slot];
    void* const zs = c->Za[slot];
    // in: not before the kernels of the slot's previous call have read it
    if (c->a_used[slot]) TPMLP_CUDA(c, cudaStreamWaitEvent(c->s_in, c->a_xfree[slot], 0));
    TPMLP_CUDA(c, cudaMemcpyAsync(xs, X_host, xbytes, cudaMemcpyHostToDevice, c->s_in));
    TPMLP_CUDA(c, cudaEventRecord(c->a_in[slot], c->s_in));
    // kernels: after the input has arrived and the slot's previous output has been copied out
    TPMLP_CUDA(c, cudaStreamWaitEvent(s, c->a_in[slot], 0));
    if (c->a_used[slot]) TPMLP_CUDA(c, cudaStreamWaitEvent(s, c->a_zfree[slot], 0));
    c->a_used[slot] = true;  // from here on the slot's events belong to this call
    ++c->a_calls;
    if (layer) {
        // the residual add of the second GEMM reads the input slot too
        if ((rc = run_layernorm(c, xs, M, c->Xn, s)) || (rc = run_gemm1(c, c->Xn, M, c->Y, s)) ||
            (rc = run_gemm2(c, c->Y, M, zs, s, xs)))
            return rc;
        TPMLP_CUDA(c, cudaEventRecord(c->a_xfree[slot], s));
    } else {
        if ((rc = run_gemm1(c, xs, M, c->Y, s))) return rc;
        TPMLP_CUDA(c, cudaEventRecord(c->a_xfree[slot], s));
        if ((rc = run_gemm2(c, c->Y, M, zs, s))) return rc;
    }
    TPMLP_CUDA(c, cudaEventRecord(c->a_zready[slot], s));
    // out: as soon as this call's second GEMM is done
    TPMLP_CUDA(c, cudaStreamWaitEvent(c->s_out, c->a_zready[slot], 0));
    TPMLP_CUDA(c, cudaMemcpyAsync(Z_host, zs, zbytes, cudaMemcpyDeviceToHost, c->s_out));
    TPMLP_CUDA(c, cudaEventRecord(c->a_zfree[slot], c->s_out));
    return TPMLP_OK;
}

int create_context(tpmlp_ctx** out, int64_t H, int64_t F, int32_t k, uint32_t flags, int kind);

// bf16 [rows][cols] map with a 64 x 64 box: an M-contiguous operand of a weight-gradient GEMM
// (inner index = output row or column, outer index = token). ld: row pitch in elements
// (0: cols).
int token_major_map(tpmlp_ctx* c, CUtensorMap* map, const void* ptr, int64_t tokens, int64_t cols,
                    int64_t ld = 0) {
    const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(tokens)};
    const uint64_t strides[1] = {static_cast<uint64_t>(ld ? ld : cols) * 2};
    const uint32_t box[2] = {64, 64};
    return encode_map(c, map, ptr, 2, dims, strides, box);
}

// fp32 out[R][C] = sum over tokens of Aop[t][r] * Bop[t][c]  (A = X or Y, B = dA or dZ);
// ldb: row pitch of Bop in elements (0: C).
int run_weight_grad(tpmlp_ctx* c, const void* Aop, int64_t R, const void* Bop, int64_t C,
                    int64_t tokens, float* out, cudaStream_t s, int64_t ldb = 0) {
    CUtensorMap ta, tb;
    int rc = token_major_map(c, &ta, Aop, tokens, R);
    if (rc || (rc = token_major_map(c, &tb, Bop, tokens, C, ldb))) return rc;
    const int bn = pick_bn(C);
    const bool pair = bn == 256 && !(c->flags & TPMLP_FLAG_SINGLE_SM);
    GemmArgs a{};
    a.M = static_cast<int>(R);
    a.ldo = static_cast<int>(C);
    a.f = static_cast<int>(C);
    a.k = 1;
    a.k2 = 1;
    a.kb_tile = static_cast<int>((tokens + tpmlp::kBK - 1) / tpmlp::kBK);
    a.kb_shard = a.kb_tile;
    const int bm = pair ? tpmlp::kPairBM : tpmlp::kBM;
    a.m_blocks = static_cast<int>((R + bm - 1) / bm);
    a.n_blocks = static_cast<int>(C / bn);
    a.num_tiles = a.m_blocks * a.n_blocks;
    a.group_m = 8;
    a.out = out;
    a.status = c->status;
    if (pair)
        return launch_pair<TPMLP_PAIR_STAGES, TPMLP_PAIR_ACC, Mode::kWeightGrad, true, true>(c, ta, tb,
                                                                                             a, s);
    switch (bn) {
        case 256: return launch_gemm<256, TPMLP_STAGES_256, Mode::kWeightGrad, true, true>(c, ta, tb, a, s);
        case 128: return launch_gemm<128, 6, Mode::kWeightGrad, true, true>(c, ta, tb, a, s);
        default: return launch_gemm<64, 8, Mode::kWeightGrad, true, true>(c, ta, tb, a, s);
    }
}

// out[c] = sum over the M rows of in[m][c] (bf16 in, row pitch ld elements (0: C), fp32 out),
// deterministic.
int run_colsum(tpmlp_ctx* c, const void* in, int64_t M, int64_t C, float* out, cudaStream_t s,
               int64_t ld = 0) {
    const int splits = static_cast<int>(std::min<int64_t>((M + 255) / 256, 128));
    const int rows_per_split = static_cast<int>((M + splits - 1) / splits);
    const int64_t need = static_cast<int64_t>(splits) * C;
    if (need > c->colsum_floats) {
        TPMLP_CUDA(c, cudaDeviceSynchronize());
        cudaFree(c->colsum);
        c->colsum = nullptr;
        c->colsum_floats = 0;
        TPMLP_CUDA(c, cudaMalloc(&c->colsum, static_cast<size_t>(need) * 4));
        c->colsum_floats = need;
    }
    dim3 grid(static_cast<unsigned>(C / 64), static_cast<unsigned>(splits));
    tpmlp::colsum_partial_kernel<<<grid, tpmlp::kColsumThreads, 0, s>>>(
        static_cast<const uint16_t*>(in), static_cast<int>(M), static_cast<int>(C),
        static_cast<int>(ld ? ld : C), rows_per_split, c->colsum);
    TPMLP_CUDA(c, cudaGetLastError());
    tpmlp::colsum_final_kernel<<<static_cast<unsigned>((C + 255) / 256), 256, 0, s>>>(
        c->colsum, splits, static_cast<int>(C), out);
    TPMLP_CUDA(c, cudaGetLastError());
    c->launches += 2;
    return TPMLP_OK;
}

}  // namespace

extern "C" {

int tpmlp_create(tpmlp_ctx** out, int64_t H, int64_t F, int32_t k, uint32_t flags) {
    if (!out) return TPMLP_ERR_INVALID_ARG;
    *out = nullptr;
    if (H <= 0 || F <= 0 || k <= 0) return TPMLP_ERR_INVALID_ARG;
    if (flags & ~(TPMLP_FLAG_Z_FP32 | TPMLP_FLAG_SINGLE_SM | TPMLP_FLAG_SWIGLU |
                  TPMLP_FLAG_FIXED_ORDER))
        return TPMLP_ERR_INVALID_ARG;
    if (H % 64 || F % 64 || F % k || (F / k) % 64) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    if (H > (int64_t(1) << 20) || F > (int64_t(1) << 22)) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    return create_context(out, H, F, k, flags, kKindBlock);
}

int tpmlp_linear_create(tpmlp_ctx** out, int32_t kind, int64_t K, int64_t N, int32_t k,
                        uint32_t flags) {
    if (!out) return TPMLP_ERR_INVALID_ARG;
    *out = nullptr;
    if (K <= 0 || N <= 0 || k <= 0) return TPMLP_ERR_INVALID_ARG;
    if (kind != TPMLP_LINEAR_COLUMN && kind != TPMLP_LINEAR_ROW) return TPMLP_ERR_INVALID_ARG;
    if (flags & ~(TPMLP_FLAG_Z_FP32 | TPMLP_FLAG_SINGLE_SM | TPMLP_FLAG_FIXED_ORDER))
        return TPMLP_ERR_INVALID_ARG;
    const int64_t split = (kind == TPMLP_LINEAR_COLUMN) ? N : K;  // the sharded dimension
    if (K % 64 || N % 64 || split % k || (split / k) % 64) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    if (K > (int64_t(1) << 22) || N > (int64_t(1) << 22)) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    // column: the first GEMM's roles (reduction H := K, outputs F := N);
    // row:    the second GEMM's roles (reduction F := K, outputs H := N)
    if (kind == TPMLP_LINEAR_COLUMN) return create_context(out, K, N, k, flags, kKindColumn);
    return create_context(out, N, K, k, flags, kKindRow);
}

}  // extern "C"

namespace {

int create_context(tpmlp_ctx** out, int64_t H, int64_t F, int32_t k, uint32_t flags, int kind) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TPMLP_ERR_CUDA;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return TPMLP_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return TPMLP_ERR_ARCH;

    tpmlp_ctx* c = new (std::nothrow) tpmlp_ctx();
    if (!c) return TPMLP_ERR_OOM;
    c->device = dev;
    c->num_sms = prop.multiProcessorCount;
    {
        // the planners' rates from the device's SM count, clock and memory system (an
        // attribute that cannot be read counts as not reported: 0)
        int sm_khz = 0, mem_khz = 0, bus_bits = 0;
        if (cudaDeviceGetAttribute(&sm_khz, cudaDevAttrClockRate, dev) != cudaSuccess) sm_khz = 0;
        if (cudaDeviceGetAttribute(&mem_khz, cudaDevAttrMemoryClockRate, dev) != cudaSuccess) mem_khz = 0;
        if (cudaDeviceGetAttribute(&bus_bits, cudaDevAttrGlobalMemoryBusWidth, dev) != cudaSuccess)
            bus_bits = 0;
        cudaGetLastError();
        c->rates = tpmlp::device_rates(c->num_sms, sm_khz, mem_khz, bus_bits);
    }
    c->H = H;
    c->F = F;
    c->k = k;
    c->f = F / k;
    c->flags = flags;
    c->kind = kind;
    c->gated = (flags & TPMLP_FLAG_SWIGLU) != 0;
    // gated: each first-GEMM tile holds G gate + G up columns of the same G outputs
    c->gate_block = (c->f % 128 == 0) ? 128 : 64;
    c->bn1 = c->gated ? 2 * c->gate_block : pick_bn(c->f);
    c->bn2 = pick_bn(H);
    // 256 x 256 tiles on CTA pairs wherever the output width allows it
    c->pair1 = c->bn1 == 256 && !(flags & TPMLP_FLAG_SINGLE_SM);
    c->pair2 = c->bn2 == 256 && !(flags & TPMLP_FLAG_SINGLE_SM);
    int rc = TPMLP_OK;
    cudaError_t e;
    const size_t parts1 = c->gated ? 2 : 1;  // gate and up packed together
    const bool first = kind != kKindRow, second = kind != kKindColumn;
    if ((first && (e = cudaMalloc(&c->W1p, parts1 * H * F * 2)) != cudaSuccess) ||
        (second && (e = cudaMalloc(&c->W2p, static_cast<size_t>(H) * F * 2)) != cudaSuccess) ||
        (first && (e = cudaMalloc(&c->b1, parts1 * F * 4)) != cudaSuccess) ||
        (second && (e = cudaMalloc(&c->b2, static_cast<size_t>(H) * 4)) != cudaSuccess) ||
        (e = cudaMalloc(&c->status, sizeof(int))) != cudaSuccess ||
        (e = cudaMemset(c->status, 0, sizeof(int))) != cudaSuccess) {
        rc = (e == cudaErrorMemoryAllocation) ? TPMLP_ERR_OOM : TPMLP_ERR_CUDA;
        tpmlp_destroy(c);
        return rc;
    }
    // workspace of the split reduction: two 256 KB slots per CTA pair, 16 counters per tile
    const size_t pairs = static_cast<size_t>(c->num_sms / 2);
    const size_t ncount = static_cast<size_t>(c->num_sms) * 2 * tpmlp::kEpiWarps;
    if (!(flags & (TPMLP_FLAG_SINGLE_SM | TPMLP_FLAG_FIXED_ORDER)) &&
        ((e = cudaMalloc(&c->sk_partial, pairs * 4 * tpmlp::kSkSlotFloats * sizeof(float))) != cudaSuccess ||
         (e = cudaMalloc(&c->sk_count, ncount * sizeof(uint32_t))) != cudaSuccess ||
         (e = cudaMemset(c->sk_count, 0, ncount * sizeof(uint32_t))) != cudaSuccess)) {
        rc = (e == cudaErrorMemoryAllocation) ? TPMLP_ERR_OOM : TPMLP_ERR_CUDA;
        tpmlp_destroy(c);
        return rc;
    }
    *out = c;
    return TPMLP_OK;
}

}  // namespace

extern "C" {

int tpmlp_pack_shards(tpmlp_ctx* c, const void* W1, const void* b1, const void* W2, const void* b2,
                      void* stream) {
    if (!c || !W1 || !b1 || !W2 || !b2 || c->gated || c->kind != kKindBlock)
        return TPMLP_ERR_INVALID_ARG;
    if (int rc = check_device(c)) return rc;
    if (!aligned16(W1) || !aligned16(W2) || (reinterpret_cast<uintptr_t>(b1) & 1) ||
        (reinterpret_cast<uintptr_t>(b2) & 1))
        return TPMLP_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int T = tpmlp::kTransposeTile;
    c->packed = false;
    {
        // W1 [H][F] -> W1p [F][H] (= [k][f][H]: shard i is rows [i f, (i+1) f))
        dim3 grid(static_cast<unsigned>(c->F / T), static_cast<unsigned>(c->H / T), 1);
        tpmlp::transpose_bf16_kernel<<<grid, dim3(64, 4), 0, s>>>(
            static_cast<const uint16_t*>(W1), c->W1p, static_cast<int>(c->H),
            static_cast<int>(c->F), 0, 0);
        TPMLP_CUDA(c, cudaGetLastError());
        ++c->launches;
    }
    tpmlp::bf16_to_f32_kernel<<<static_cast<unsigned>((c->F + 255) / 256), 256, 0, s>>>(
        static_cast<const uint16_t*>(b1), c->b1, c->F);
    TPMLP_CUDA(c, cudaGetLastError());
    ++c->launches;
    int rc = pack_second_layer(c, W2, b2, s);
    if (rc) return rc;
    if ((rc = encode_weight_maps(c))) return rc;
    c->packed = true;
    return TPMLP_OK;
}

int tpmlp_pack_shards_swiglu(tpmlp_ctx* c, const void* Wg, const void* bg, const void* Wu,
                             const void* bu, const void* W2, const void* b2, void* stream) {
    if (!c || !Wg || !bg || !Wu || !bu || !W2 || !b2 || !c->gated || c->kind != kKindBlock)
        return TPMLP_ERR_INVALID_ARG;
    if (int rc = check_device(c)) return rc;
    if (!aligned16(Wg) || !aligned16(Wu) || !aligned16(W2) ||
        ((reinterpret_cast<uintptr_t>(bg) | reinterpret_cast<uintptr_t>(bu) |
          reinterpret_cast<uintptr_t>(b2)) & 1))
        return TPMLP_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int T = tpmlp::kTransposeTile;
    c->packed = false;
    const void* parts[2] = {Wg, Wu};
    const void* biases[2] = {bg, bu};
    for (int part = 0; part < 2; ++part) {
        // gate (part 0) / up (part 1) [H][F] -> interleaved rows of W1p [k][2f][H]
        dim3 grid(static_cast<unsigned>(c->F / T), static_cast<unsigned>(c->H / T), 1);
        tpmlp::transpose_interleave_bf16_kernel<<<grid, dim3(64, 4), 0, s>>>(
            static_cast<const uint16_t*>(parts[part]), c->W1p, static_cast<int>(c->H),
            static_cast<int>(c->F), c->gate_block, part);
        TPMLP_CUDA(c, cudaGetLastError());
        tpmlp::interleave_bias_kernel<<<static_cast<unsigned>((c->F + 255) / 256), 256, 0, s>>>(
            static_cast<const uint16_t*>(biases[part]), c->b1, static_cast<int>(c->F),
            c->gate_block, part);
        TPMLP_CUDA(c, cudaGetLastError());
        c->launches += 2;
    }
    int rc = pack_second_layer(c, W2, b2, s);
    if (rc) return rc;
    if ((rc = encode_weight_maps(c))) return rc;
    c->packed = true;
    return TPMLP_OK;
}

int tpmlp_reserve(tpmlp_ctx* c, int64_t max_tokens) {
    if (!c || c->kind != kKindBlock || max_tokens < 0) return TPMLP_ERR_INVALID_ARG;
    if (int rc = check_device(c)) return rc;
    if (max_tokens > (int64_t(1) << 31)) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    return ensure_y(c, max_tokens);
}

int tpmlp_gemm1(tpmlp_ctx* c, const void* X, int64_t M, void* Y, void* stream) {
    int rc = check_ctx(c);
    if (rc) return rc;
    if (M < 0) return TPMLP_ERR_INVALID_ARG;
    if (M == 0) return TPMLP_OK;
    if (!X || !Y) return TPMLP_ERR_INVALID_ARG;
    if (M > (int64_t(1) << 31)) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(X) || !aligned16(Y)) return TPMLP_ERR_MISALIGNED;
    return run_gemm1(c, X, M, Y, static_cast<cudaStream_t>(stream));
}

int tpmlp_gemm2(tpmlp_ctx* c, const void* Y, int64_t M, void* Z, void* stream) {
    int rc = check_ctx(c);
    if (rc) return rc;
    if (M < 0) return TPMLP_ERR_INVALID_ARG;
    if (M == 0) return TPMLP_OK;
    if (!Y || !Z) return TPMLP_ERR_INVALID_ARG;
    if (M > (int64_t(1) << 31)) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(Y) || !aligned16(Z)) return TPMLP_ERR_MISALIGNED;
    return run_gemm2(c, Y, M, Z, static_cast<cudaStream_t>(stream));
}

int tpmlp_forward_marked(tpmlp_ctx* c, const void* X, int64_t B, int64_t S, void* Z,
                         void* after_gemm1, void* stream) {
    int rc = check_ctx(c);
    if (rc) return rc;
    if ((rc = check_tokens(B, S))) return rc;
    const int64_t M = B * S;
    if (M == 0) return TPMLP_OK;
    if (!X || !Z || !after_gemm1) return TPMLP_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Z)) return TPMLP_ERR_MISALIGNED;
    if ((rc = ensure_y(c, M))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((rc = run_gemm1(c, X, M, c->Y, s))) return rc;
    TPMLP_CUDA(c, cudaEventRecord(static_cast<cudaEvent_t>(after_gemm1), s));
    return run_gemm2(c, c->Y, M, Z, s);
}

int tpmlp_forward(tpmlp_ctx* c, const void* X, int64_t B, int64_t S, void* Z, void* stream) {
    int rc = check_ctx(c);
    if (rc) return rc;
    if ((rc = check_tokens(B, S))) return rc;
    const int64_t M = B * S;
    if (M == 0) return TPMLP_OK;
    if (!X || !Z) return TPMLP_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Z)) return TPMLP_ERR_MISALIGNED;
    if ((rc = ensure_y(c, M))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((rc = run_gemm1(c, X, M, c->Y, s))) return rc;
    return run_gemm2(c, c->Y, M, Z, s);
}

int tpmlp_forward_host(tpmlp_ctx* c, const void* X_host, int64_t B, int64_t S, void* Z_host,
                       void* stream) {
    return run_host_pipeline(c, X_host, B, S, Z_host, static_cast<cudaStream_t>(stream), false);
}

int tpmlp_forward_host_async(tpmlp_ctx* c, const void* X_host, int64_t B, int64_t S,
                             void* Z_host, void* stream) {
    return run_host_async(c, X_host, B, S, Z_host, static_cast<cudaStream_t>(stream), false);
}

int tpmlp_host_wait(tpmlp_ctx* c) {
    if (!c) return TPMLP_ERR_INVALID_ARG;
    if (int rc = check_device(c)) return rc;
    if (!c->s_in || !c->s_out) return TPMLP_OK;  // no host-buffer call has queued work
    // every output copy waits for its call's kernels, which wait for its input copy
    TPMLP_CUDA(c, cudaStreamSynchronize(c->s_out));
    TPMLP_CUDA(c, cudaStreamSynchronize(c->s_in));
    return TPMLP_OK;
}

int tpmlp_set_layernorm(tpmlp_ctx* c, const void* gamma, const void* beta, float eps,
                        void* stream) {
    // the block's input, or a column-parallel layer's input (LayerNorm before Q/K/V)
    if (!c || !gamma || !beta || c->kind == kKindRow) return TPMLP_ERR_INVALID_ARG;
    if (int rc = check_device(c)) return rc;
    if (!(eps >= 0.0f) || eps > 1.0f) return TPMLP_ERR_INVALID_ARG;  // also rejects NaN
    if (c->H > tpmlp::kNormMaxH) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    if ((reinterpret_cast<uintptr_t>(gamma) | reinterpret_cast<uintptr_t>(beta)) & 1)
        return TPMLP_ERR_MISALIGNED;
    if (!c->ln_gamma) {
        TPMLP_CUDA(c, cudaMalloc(&c->ln_gamma, static_cast<size_t>(c->H) * 4));
        TPMLP_CUDA(c, cudaMalloc(&c->ln_beta, static_cast<size_t>(c->H) * 4));
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const unsigned blocks = static_cast<unsigned>((c->H + 255) / 256);
    tpmlp::bf16_to_f32_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint16_t*>(gamma),
                                                     c->ln_gamma, c->H);
    TPMLP_CUDA(c, cudaGetLastError());
    tpmlp::bf16_to_f32_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint16_t*>(beta),
                                                     c->ln_beta, c->H);
    TPMLP_CUDA(c, cudaGetLastError());
    c->launches += 2;
    c->ln_eps = eps;
    c->ln_set = true;
    return TPMLP_OK;
}

int tpmlp_layernorm(tpmlp_ctx* c, const void* X, int64_t M, void* Xn, void* stream) {
    if (!c || M < 0) return TPMLP_ERR_INVALID_ARG;
    if (int rc = check_device(c)) return rc;
    if (!c->ln_set) {
        c->last_error = "LayerNorm parameters not set (tpmlp_set_layernorm)";
        return TPMLP_ERR_NOT_PACKED;
    }
    if (M == 0) return TPMLP_OK;
    if (!X || !Xn) return TPMLP_ERR_INVALID_ARG;
    if (M > (int64_t(1) << 31) - 1) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(X) || !aligned16(Xn)) return TPMLP_ERR_MISALIGNED;
    return run_layernorm(c, X, M, Xn, static_cast<cudaStream_t>(stream));
}

int tpmlp_block_forward(tpmlp_ctx* c, const void* X, int64_t B, int64_t S, void* Z,
                        void* stream) {
    int rc = check_ctx(c);
    if (rc) return rc;
    if (!c->ln_set) {
        c->last_error = "LayerNorm parameters not set (tpmlp_set_layernorm)";
        return TPMLP_ERR_NOT_PACKED;
    }
    if ((rc = check_tokens(B, S))) return rc;
    const int64_t M = B * S;
    if (M == 0) return TPMLP_OK;
    if (!X || !Z) return TPMLP_ERR_INVALID_ARG;
    if (M > (int64_t(1) << 31) - 1) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(X) || !aligned16(Z)) return TPMLP_ERR_MISALIGNED;
    if ((rc = ensure_xn(c, M)) || (rc = ensure_y(c, M))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((rc = run_layernorm(c, X, M, c->Xn, s))) return rc;
    if ((rc = run_gemm1(c, c->Xn, M, c->Y, s))) return rc;
    return run_gemm2(c, c->Y, M, Z, s, X);  // epilogue: Z = X + (Y W2 + b2)
}

int tpmlp_block_forward_marked(tpmlp_ctx* c, const void* X, int64_t B, int64_t S, void* Z,
                               void* after_layernorm, void* after_gemm1, void* stream) {
    int rc = check_ctx(c);
    if (rc) return rc;
    if (!c->ln_set) {
        c->last_error = "LayerNorm parameters not set (tpmlp_set_layernorm)";
        return TPMLP_ERR_NOT_PACKED;
    }
    if ((rc = check_tokens(B, S))) return rc;
    const int64_t M = B * S;
    if (M == 0) return TPMLP_OK;
    if (!X || !Z || !after_layernorm || !after_gemm1) return TPMLP_ERR_INVALID_ARG;
    if (M > (int64_t(1) << 31) - 1) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(X) || !aligned16(Z)) return TPMLP_ERR_MISALIGNED;
    if ((rc = ensure_xn(c, M)) || (rc = ensure_y(c, M))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((rc = run_layernorm(c, X, M, c->Xn, s))) return rc;
    TPMLP_CUDA(c, cudaEventRecord(static_cast<cudaEvent_t>(after_layernorm), s));
    if ((rc = run_gemm1(c, c->Xn, M, c->Y, s))) return rc;
    TPMLP_CUDA(c, cudaEventRecord(static_cast<cudaEvent_t>(after_gemm1), s));
    return run_gemm2(c, c->Y, M, Z, s, X);
}

int tpmlp_block_forward_host(tpmlp_ctx* c, const void* X_host, int64_t B, int64_t S,
                             void* Z_host, void* stream) {
    return run_host_pipeline(c, X_host, B, S, Z_host, static_cast<cudaStream_t>(stream), true);
}

int tpmlp_block_forward_host_async(tpmlp_ctx* c, const void* X_host, int64_t B, int64_t S,
                                   void* Z_host, void* stream) {
    return run_host_async(c, X_host, B, S, Z_host, static_cast<cudaStream_t>(stream), true);
}

int tpmlp_gemm2_residual(tpmlp_ctx* c, const void* Y, int64_t M, void* Z, const void* R,
                         void* stream) {
    int rc = check_ctx(c);
    if (rc) return rc;
    if (M < 0) return TPMLP_ERR_INVALID_ARG;
    if (M == 0) return TPMLP_OK;
    if (!Y || !Z || !R) return TPMLP_ERR_INVALID_ARG;
    if (M > (int64_t(1) << 31)) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(Y) || !aligned16(Z) || !aligned16(R)) return TPMLP_ERR_MISALIGNED;
    return run_gemm2(c, Y, M, Z, static_cast<cudaStream_t>(stream), R);
}

int tpmlp_linear_pack(tpmlp_ctx* c, const void* W, const void* b, void* stream) {
    if (!c || !W || !b || c->kind == kKindBlock) return TPMLP_ERR_INVALID_ARG;
    if (int rc = check_device(c)) return rc;
    if (!aligned16(W) || (reinterpret_cast<uintptr_t>(b) & 1)) return TPMLP_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    c->packed = false;
    int rc = TPMLP_OK;
    if (c->kind == kKindColumn) {
        // W [K = H][N = F] -> W1p [F][H] (= [k][f][H]), the layout of the first GEMM
        const int T = tpmlp::kTransposeTile;
        dim3 grid(static_cast<unsigned>(c->F / T), static_cast<unsigned>(c->H / T), 1);
        tpmlp::transpose_bf16_kernel<<<grid, dim3(64, 4), 0, s>>>(
            static_cast<const uint16_t*>(W), c->W1p, static_cast<int>(c->H),
            static_cast<int>(c->F), 0, 0);
        TPMLP_CUDA(c, cudaGetLastError());
        tpmlp::bf16_to_f32_kernel<<<static_cast<unsigned>((c->F + 255) / 256), 256, 0, s>>>(
            static_cast<const uint16_t*>(b), c->b1, c->F);
        TPMLP_CUDA(c, cudaGetLastError());
        c->launches += 2;
    } else {
        // W [K = F][N = H] -> W2p [k][H][f], the layout of the second GEMM
        if ((rc = pack_second_layer(c, W, b, s))) return rc;
    }
    if ((rc = encode_weight_maps(c))) return rc;
    c->packed = true;
    return TPMLP_OK;
}

int tpmlp_linear_forward(tpmlp_ctx* c, const void* X, int64_t M, void* out, void* stream) {
    if (!c || c->kind == kKindBlock || M < 0) return TPMLP_ERR_INVALID_ARG;
    if (int rc = check_device(c)) return rc;
    if (!c->packed) return TPMLP_ERR_NOT_PACKED;
    if (M == 0) return TPMLP_OK;
    if (!X || !out) return TPMLP_ERR_INVALID_ARG;
    if (M > (int64_t(1) << 31) - 1) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(X) || !aligned16(out)) return TPMLP_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (c->kind == kKindColumn) return run_gemm1(c, X, M, out, s, /*linear=*/true);
    return run_gemm2(c, X, M, out, s);
}

int tpmlp_forward_train(tpmlp_ctx* c, const void* X, int64_t B, int64_t S, void* Z, void* Ysave,
                        void* Asave, void* stream) {
    int rc = check_ctx(c);
    if (rc) return rc;
    if ((rc = check_tokens(B, S))) return rc;
    const int64_t M = B * S;
    if (M == 0) return TPMLP_OK;
    if (!X || !Z || !Ysave || !Asave) return TPMLP_ERR_INVALID_ARG;
    if (M > (int64_t(1) << 31) - 1) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(X) || !aligned16(Z) || !aligned16(Ysave) || !aligned16(Asave))
        return TPMLP_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((rc = run_gemm1(c, X, M, Ysave, s, false, Asave))) return rc;
    return run_gemm2(c, Ysave, M, Z, s);
}

int tpmlp_backward(tpmlp_ctx* c, const void* dZ, const void* X, const void* Ysave,
                   const void* Asave, const void* W1, const void* W2, int64_t B, int64_t S,
                   void* dX, void* dW1, void* db1, void* dW2, void* db2, void* stream) {
    int rc = check_ctx(c);
    if (rc) return rc;
    if (c->gated) return TPMLP_ERR_INVALID_ARG;
    if ((rc = check_tokens(B, S))) return rc;
    const int64_t M = B * S;
    if (M == 0) return TPMLP_OK;
    if (!dZ || !X || !Ysave || !Asave || !W1 || !W2 || !dX || !dW1 || !db1 || !dW2 || !db2)
        return TPMLP_ERR_INVALID_ARG;
    if (M > (int64_t(1) << 31) - 1) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    for (const void* p : {dZ, X, Ysave, Asave, W1, W2, static_cast<const void*>(dX),
                          static_cast<const void*>(dW1), static_cast<const void*>(db1),
                          static_cast<const void*>(dW2), static_cast<const void*>(db2)})
        if (!aligned16(p)) return TPMLP_ERR_MISALIGNED;
    if ((rc = ensure_y(c, M))) return rc;  // the context's Y buffer holds dA
    if (!c->zeros) {
        const size_t n = static_cast<size_t>(std::max(c->H, c->F));
        TPMLP_CUDA(c, cudaMalloc(&c->zeros, n * 4));
        TPMLP_CUDA(c, cudaMemset(c->zeros, 0, n * 4));
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // (1) dA = (dZ W2^T) * GeLU'(A): the first GEMM's tiling over the caller's W2 [F][H],
    //     whose row shards are K-major blocks [k][f][H]
    {
        CUtensorMap tdz, tw2, tw2p;
        int r = activation_map(c, dZ, M, c->H, c->x_map_ptr, c->x_map_rows, c->tmX);
        if (r) return r;
        tdz = c->tmX;
        const uint64_t dims[3] = {static_cast<uint64_t>(c->H), static_cast<uint64_t>(c->f),
                                  static_cast<uint64_t>(c->k)};
        const uint64_t strides[2] = {static_cast<uint64_t>(c->H) * 2,
                                     static_cast<uint64_t>(c->f) * c->H * 2};
        const uint32_t box[3] = {tpmlp::kBK, static_cast<uint32_t>(c->bn1), 1};
        const uint32_t box_pair[3] = {tpmlp::kBK, 128, 1};
        if ((r = encode_map(c, &tw2, W2, 3, dims, strides, box)) ||
            (r = encode_map(c, &tw2p, W2, 3, dims, strides, box_pair)))
            return r;
        GemmArgs a = base_args(c, M, static_cast<int>(c->F), c->pair1 ? tpmlp::kPairBM : tpmlp::kBM,
                               c->pair1 ? tpmlp::kPairBN : c->bn1, TPMLP_GROUP_M1);
        a.kb_tile = static_cast<int>(c->H / tpmlp::kBK);
        a.kb_shard = a.kb_tile;
        a.out = c->Y;
        a.residual = Asave;
        r = c->pair1 ? launch_pair<TPMLP_PAIR_STAGES, TPMLP_PAIR_ACC, Mode::kBwdDA, false>(c, tdz, tw2p, a, s)
                     : dispatch_gemm<Mode::kBwdDA, false>(c, c->bn1, tdz, tw2, a, s);
        if (r) return r;
    }
    // (2) dX = sum_i dA_i W1_i^T: the second GEMM's shard-major reduction over the caller's
    //     W1 [H][F], read as [k][H][f] blocks (element (j, h, i) at W1 + h F + i f + j)
    {
        CUtensorMap tw1, tw1p;
        const uint64_t dims[3] = {static_cast<uint64_t>(c->f), static_cast<uint64_t>(c->H),
                                  static_cast<uint64_t>(c->k)};
        const uint64_t strides[2] = {static_cast<uint64_t>(c->F) * 2, static_cast<uint64_t>(c->f) * 2};
        const uint32_t box[3] = {tpmlp::kBK, static_cast<uint32_t>(c->bn2), 1};
        const uint32_t box_pair[3] = {tpmlp::kBK, 128, 1};
        int r = encode_map(c, &tw1, W1, 3, dims, strides, box);
        if (r || (r = encode_map(c, &tw1p, W1, 3, dims, strides, box_pair))) return r;
        if ((r = activation_map(c, c->Y, M, c->F, c->y_map_ptr, c->y_map_rows, c->tmY))) return r;
        GemmArgs a = base_args(c, M, static_cast<int>(c->H), c->pair2 ? tpmlp::kPairBM : tpmlp::kBM,
                               c->pair2 ? tpmlp::kPairBN : c->bn2, TPMLP_GROUP_M2);
        a.kb_shard = static_cast<int>(c->f / tpmlp::kBK);
        a.kb_tile = a.kb_shard * c->k;
        a.bias = c->zeros;
        a.out = dX;
        const bool f32 = (c->flags & TPMLP_FLAG_Z_FP32) != 0;
        if (c->pair2)
            r = f32 ? launch_gemm2_pair<Mode::kGemm2, true>(c, c->tmY, tw1p, a, s)
                    : launch_gemm2_pair<Mode::kGemm2, false>(c, c->tmY, tw1p, a, s);
        else
            r = f32 ? dispatch_gemm<Mode::kGemm2, true>(c, c->bn2, c->tmY, tw1, a, s)
                    : dispatch_gemm<Mode::kGemm2, false>(c, c->bn2, c->tmY, tw1, a, s);
        if (r) return r;
    }
    // (3) dW1 = X^T dA [H][F], (4) dW2 = Y^T dZ [F][H]: reductions over the tokens
    if ((rc = run_weight_grad(c, X, c->H, c->Y, c->F, M, static_cast<float*>(dW1), s))) return rc;
    if ((rc = run_weight_grad(c, Ysave, c->F, dZ, c->H, M, static_cast<float*>(dW2), s))) return rc;
    // (5) db1 = sum over tokens of dA, db2 = sum over tokens of dZ
    if ((rc = run_colsum(c, c->Y, M, c->F, static_cast<float*>(db1), s))) return rc;
    return run_colsum(c, dZ, M, c->H, static_cast<float*>(db2), s);
}

int tpmlp_backward_swiglu(tpmlp_ctx* c, const void* dZ, const void* X, const void* Ysave,
                          const void* Asave, const void* Wg, const void* Wu, const void* W2,
                          int64_t B, int64_t S, void* dX, void* dWg, void* dbg, void* dWu,
                          void* dbu, void* dW2, void* db2, void* stream) {
    int rc = check_ctx(c);
    if (rc) return rc;
    if (!c->gated) return TPMLP_ERR_INVALID_ARG;
    if ((rc = check_tokens(B, S))) return rc;
    const int64_t M = B * S;
    if (M == 0) return TPMLP_OK;
    if (!dZ || !X || !Ysave || !Asave || !Wg || !Wu || !W2 || !dX || !dWg || !dbg || !dWu ||
        !dbu || !dW2 || !db2)
        return TPMLP_ERR_INVALID_ARG;
    if (M > (int64_t(1) << 31) - 1) return TPMLP_ERR_UNSUPPORTED_SHAPE;
    for (const void* p : {dZ, X, Ysave, Asave, Wg, Wu, W2, static_cast<const void*>(dX),
                          static_cast<const void*>(dWg), static_cast<const void*>(dbg),
                          static_cast<const void*>(dWu), static_cast<const void*>(dbu),
                          static_cast<const void*>(dW2), static_cast<const void*>(db2)})
        if (!aligned16(p)) return TPMLP_ERR_MISALIGNED;
    const int64_t F = c->F, H = c->H, f = c->f;
    // dG and dU, [M][2F] (dU from column F on), in the context's gradient buffer
    if (M * 2 * F > c->dgu_elems) {
        TPMLP_CUDA(c, cudaDeviceSynchronize());  // the old buffer may still be in use
        cudaFree(c->dgu);
        c->dgu = nullptr;
        c->dgu_elems = 0;
        const int64_t rows = ((M + tpmlp::kBM - 1) / tpmlp::kBM) * tpmlp::kBM;
        TPMLP_CUDA(c, cudaMalloc(&c->dgu, static_cast<size_t>(rows * 2 * F) * 2));
        c->dgu_elems = rows * 2 * F;
    }
    if (!c->zeros) {
        const size_t n = static_cast<size_t>(std::max(H, F));
        TPMLP_CUDA(c, cudaMalloc(&c->zeros, n * 4));
        TPMLP_CUDA(c, cudaMemset(c->zeros, 0, n * 4));
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The non-gated context's tile choices: the pair kernel where the output width allows.
    const bool single = (c->flags & TPMLP_FLAG_SINGLE_SM) != 0;
    const int bn_f = pick_bn(f), bn_h = pick_bn(H);
    const bool pair_f = bn_f == 256 && !single, pair_h = bn_h == 256 && !single;

    // (1) dY = dZ W2^T per column shard of W2 [F][H] (K-major blocks [k][f][H]); the epilogue
    //     turns it into dG = dY U SiLU'(G) and dU = dY SiLU(G) with the saved G, U
    {
        CUtensorMap tdz, tw2;
        int r = activation_map(c, dZ, M, H, c->x_map_ptr, c->x_map_rows, c->tmX);
        if (r) return r;
        tdz = c->tmX;
        const uint64_t dims[3] = {static_cast<uint64_t>(H), static_cast<uint64_t>(f),
                                  static_cast<uint64_t>(c->k)};
        const uint64_t strides[2] = {static_cast<uint64_t>(H) * 2, static_cast<uint64_t>(f) * H * 2};
        const uint32_t box[3] = {tpmlp::kBK, static_cast<uint32_t>(pair_f ? 128 : bn_f), 1};
        if ((r = encode_map(c, &tw2, W2, 3, dims, strides, box))) return r;
        const int tile_n = pair_f ? tpmlp::kPairBN : bn_f;
        GemmArgs a = base_args(c, M, static_cast<int>(2 * F), pair_f ? tpmlp::kPairBM : tpmlp::kBM,
                               tile_n, TPMLP_GROUP_M1);
        a.n_blocks = static_cast<int>(F / tile_n);  // output columns [0, F); rows of pitch 2F
        a.num_tiles = a.m_blocks * a.n_blocks;
        a.kb_tile = static_cast<int>(H / tpmlp::kBK);
        a.kb_shard = a.kb_tile;
        a.out = c->dgu;
        a.residual = Asave;
        a.half = static_cast<int>(F);
        r = pair_f ? launch_pair<TPMLP_PAIR_STAGES, TPMLP_PAIR_ACC, Mode::kBwdGated, false>(c, tdz, tw2, a, s)
                   : dispatch_gemm<Mode::kBwdGated, false>(c, bn_f, tdz, tw2, a, s);
        if (r) return r;
    }
    // (2) dX = sum_i (dG_i Wg_i^T + dU_i Wu_i^T): the second GEMM's shard-major reduction over
    //     2k shards of [dG | dU] -- the gate shards read Wg [H][F] and the up shards Wu [H][F],
    //     each as [k][H][f] blocks -- all into one accumulator
    {
        CUtensorMap tdgu, twg, twu;
        const uint64_t dims[3] = {static_cast<uint64_t>(f), static_cast<uint64_t>(H),
                                  static_cast<uint64_t>(c->k)};
        const uint64_t strides[2] = {static_cast<uint64_t>(F) * 2, static_cast<uint64_t>(f) * 2};
        const uint32_t box[3] = {tpmlp::kBK, static_cast<uint32_t>(pair_h ? 128 : bn_h), 1};
        int r = encode_map(c, &twg, Wg, 3, dims, strides, box);
        if (r || (r = encode_map(c, &twu, Wu, 3, dims, strides, box))) return r;
        const uint64_t adims[2] = {static_cast<uint64_t>(2 * F), static_cast<uint64_t>(M)};
        const uint64_t astrides[1] = {static_cast<uint64_t>(2 * F) * 2};
        const uint32_t abox[2] = {tpmlp::kBK, tpmlp::kBM};
        if ((r = encode_map(c, &tdgu, c->dgu, 2, adims, astrides, abox))) return r;
        GemmArgs a = base_args(c, M, static_cast<int>(H), pair_h ? tpmlp::kPairBM : tpmlp::kBM,
                               pair_h ? tpmlp::kPairBN : bn_h, TPMLP_GROUP_M2);
        a.k = 2 * c->k;
        a.k2 = c->k;
        a.kb_shard = static_cast<int>(f / tpmlp::kBK);
        a.kb_tile = a.kb_shard * a.k;
        a.bias = c->zeros;
        a.out = dX;
        const bool f32 = (c->flags & TPMLP_FLAG_Z_FP32) != 0;
        if (pair_h)
            r = f32 ? launch_gemm2_pair<Mode::kGemm2, true>(c, tdgu, twg, a, s, &twu)
                    : launch_gemm2_pair<Mode::kGemm2, false>(c, tdgu, twg, a, s, &twu);
        else
            r = f32 ? dispatch_gemm<Mode::kGemm2, true>(c, bn_h, tdgu, twg, a, s, &twu)
                    : dispatch_gemm<Mode::kGemm2, false>(c, bn_h, tdgu, twg, a, s, &twu);
        if (r) return r;
    }
    // (3) dWg = X^T dG, dWu = X^T dU [H][F]; (4) dW2 = Y^T dZ [F][H]: reductions over tokens
    if ((rc = run_weight_grad(c, X, H, c->dgu, F, M, static_cast<float*>(dWg), s, 2 * F))) return rc;
    if ((rc = run_weight_grad(c, X, H, c->dgu + F, F, M, static_cast<float*>(dWu), s, 2 * F)))
        return rc;
    if ((rc = run_weight_grad(c, Ysave, F, dZ, H, M, static_cast<float*>(dW2), s))) return rc;
    // (5) dbg, dbu, db2: sums over tokens
    if ((rc = run_colsum(c, c->dgu, M, F, static_cast<float*>(dbg), s, 2 * F))) return rc;
    if ((rc = run_colsum(c, c->dgu + F, M, F, static_cast<float*>(dbu), s, 2 * F))) return rc;
    return run_colsum(c, dZ, M, H, static_cast<float*>(db2), s);
}

int tpmlp_get_status(tpmlp_ctx* c, void* stream, int32_t* detail) {
    if (!c) return TPMLP_ERR_INVALID_ARG;
    if (int rc = check_device(c)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    TPMLP_CUDA(c, cudaStreamSynchronize(s));
    int v = 0;
    TPMLP_CUDA(c, cudaMemcpy(&v, c->status, sizeof(int), cudaMemcpyDeviceToHost));
    TPMLP_CUDA(c, cudaMemset(c->status, 0, sizeof(int)));
    if (detail) *detail = v;
    return v ? TPMLP_ERR_DEVICE_TIMEOUT : TPMLP_OK;
}

int tpmlp_packed_buffer(const tpmlp_ctx* c, int32_t which, const void** ptr, int64_t* bytes) {
    if (!c || !ptr || !bytes) return TPMLP_ERR_INVALID_ARG;
    if (!c->packed) return TPMLP_ERR_NOT_PACKED;
    switch (which) {
        case 0:
            if (!c->W1p) return TPMLP_ERR_INVALID_ARG;
            *ptr = c->W1p; *bytes = (c->gated ? 2 : 1) * c->H * c->F * 2; return TPMLP_OK;
        case 1:
            if (!c->W2p) return TPMLP_ERR_INVALID_ARG;
            *ptr = c->W2p; *bytes = c->H * c->F * 2; return TPMLP_OK;
        case 2:
            if (!c->b1) return TPMLP_ERR_INVALID_ARG;
            *ptr = c->b1; *bytes = (c->gated ? 2 : 1) * c->F * 4; return TPMLP_OK;
        case 3:
            if (!c->b2) return TPMLP_ERR_INVALID_ARG;
            *ptr = c->b2; *bytes = c->H * 4; return TPMLP_OK;
        default: return TPMLP_ERR_INVALID_ARG;
    }
}

void tpmlp_destroy(tpmlp_ctx* c) {
    if (!c) return;
    int cur = -1;
    cudaGetDevice(&cur);
    if (c->device >= 0 && cur != c->device) cudaSetDevice(c->device);
    cudaDeviceSynchronize();
    cudaFree(c->W1p);
    cudaFree(c->W2p);
    cudaFree(c->b1);
    cudaFree(c->b2);
    cudaFree(c->Y);
    cudaFree(c->Xs);
    cudaFree(c->Zs);
    for (int i = 0; i < 2; ++i) {
        cudaFree(c->Xa[i]);
        cudaFree(c->Za[i]);
        for (cudaEvent_t e : {c->a_in[i], c->a_xfree[i], c->a_zready[i], c->a_zfree[i]})
            if (e) cudaEventDestroy(e);
    }
    for (cudaEvent_t e : c->host_ev) if (e) cudaEventDestroy(e);
    for (cudaEvent_t e : c->in_ev) if (e) cudaEventDestroy(e);
    for (cudaEvent_t e : c->out_ev) if (e) cudaEventDestroy(e);
    if (c->s_in) cudaStreamDestroy(c->s_in);
    if (c->s_out) cudaStreamDestroy(c->s_out);
    cudaFree(c->Xn);
    cudaFree(c->zeros);
    cudaFree(c->colsum);
    cudaFree(c->dgu);
    cudaFree(c->ln_gamma);
    cudaFree(c->ln_beta);
    cudaFree(c->sk_partial);
    cudaFree(c->sk_count);
    cudaFree(c->status);
    if (cur >= 0 && cur != c->device) cudaSetDevice(cur);
    delete c;
}

const char* tpmlp_strerror(int status) {
    switch (status) {
        case TPMLP_OK: return "ok";
        case TPMLP_ERR_INVALID_ARG: return "invalid argument";
        case TPMLP_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (H, F, F/k multiples of 64; F % k == 0)";
        case TPMLP_ERR_NOT_PACKED: return "weights not packed (call tpmlp_pack_shards first)";
        case TPMLP_ERR_CUDA: return "CUDA error (see tpmlp_last_error)";
        case TPMLP_ERR_OOM: return "device out of memory";
        case TPMLP_ERR_DEVICE_TIMEOUT: return "a kernel gave up waiting on a pipeline barrier";
        case TPMLP_ERR_ARCH: return "device is not sm_103 (GB300)";
        case TPMLP_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
        default: return "unknown status";
    }
}

const char* tpmlp_last_error(const tpmlp_ctx* c) { return c ? c->last_error.c_str() : ""; }

int64_t tpmlp_launch_count(const tpmlp_ctx* c) { return c ? c->launches : 0; }

int tpmlp_set_device_rates(tpmlp_ctx* c, double gemm_flops, double dram_Bps, double copy_Bps) {
    if (!c) return TPMLP_ERR_INVALID_ARG;
    for (double v : {gemm_flops, dram_Bps, copy_Bps})
        if (!(v >= 0.0) || v > 1e18) return TPMLP_ERR_INVALID_ARG;  // also rejects NaN
    if (gemm_flops > 0.0) c->rates.gemm_flops = gemm_flops;
    if (dram_Bps > 0.0) c->rates.dram_Bps = dram_Bps;
    if (copy_Bps > 0.0) c->rates.copy_Bps = copy_Bps;
    c->plan_M = -1;  // re-plan the host-buffer chunks on the next call
    return TPMLP_OK;
}

int tpmlp_get_device_rates(const tpmlp_ctx* c, double* gemm_flops, double* dram_Bps,
                           double* copy_Bps) {
    if (!c || !gemm_flops || !dram_Bps || !copy_Bps) return TPMLP_ERR_INVALID_ARG;
    *gemm_flops = c->rates.gemm_flops;
    *dram_Bps = c->rates.dram_Bps;
    *copy_Bps = c->rates.copy_Bps;
    return TPMLP_OK;
}

#ifndef TPMLP_SOURCE_HASH
#define TPMLP_SOURCE_HASH "unknown"
#endif
const char* tpmlp_build_id(void) { return TPMLP_SOURCE_HASH; }

}  // extern "C"

#ifdef TPMLP_TEST_HOOKS
// Test builds only (-DTPMLP_TEST_HOOKS): a block or linear context that holds no device
// memory, recorded as belonging to `device`, and the substitute for the current-device query.
// With them, host tests drive the argument and device checks of every entry point on a
// machine without a GPU. tpmlp_destroy releases such a context.
extern "C" TPMLP_API tpmlp_ctx* tpmlp_test_host_context(int64_t H, int64_t F, int32_t k,
                                                        int32_t device, int32_t kind,
                                                        int32_t packed, uint32_t flags) {
    tpmlp_ctx* c = new (std::nothrow) tpmlp_ctx();
    if (!c) return nullptr;
    c->flags = flags;
    c->gated = (flags & TPMLP_FLAG_SWIGLU) != 0;
    c->device = device;
    c->num_sms = 152;
    c->H = H;
    c->F = F;
    c->k = k;
    c->f = F / k;
    c->kind = kind;
    c->packed = packed != 0;
    c->rates = tpmlp::device_rates(0, 0, 0, 0);
    return c;
}

extern "C" TPMLP_API void tpmlp_test_set_current_device(int32_t device) {
    g_test_current_device.store(device);
}
#endif

// ---------------------------------------------------------------------------------------
// Allocation-free forward pass.
//
// Some callers cannot call cudaMalloc at the point where they run the block: a serving
// process that hands all free device memory to its own allocator at start-up (caches,
// memory pools) and forbids later driver allocations, or code on a latency-critical path
// where an allocation would implicitly synchronise the device. For them the intermediate
// activations Y live in one fixed device array compiled into this library instead of a
// buffer the context allocates. The array is TPMLP_NOALLOC_SCRATCH_BYTES long; every GPU
// that loads the library holds it until the process exits.
namespace {

static __device__ __align__(256) unsigned char g_noalloc_y[TPMLP_NOALLOC_SCRATCH_BYTES];

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mu;
struct NoallocSlot {
    unsigned long long ctx_id;  // the CUDA context the address was looked up in
    void* ptr;                  // device address of g_noalloc_y in that context
};
NoallocSlot g_noalloc[kNoallocMaxDevices] = {};

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_fn_once;

// The unique id of the CUDA context current on this thread (0: none current, or the driver
// cannot tell). Ids are never reused within a process, so a context created after a device
// reset gets a new one.
unsigned long long current_context_id() {
    std::call_once(g_ctx_fn_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
        cudaGetLastError();
    });
    if (!g_ctx_current || !g_ctx_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// The device address of g_noalloc_y on the context's device, which the caller has checked to
// be current. In host code the array's name is only a host-side stand-in, so the address is
// looked up (cudaGetSymbolAddress) on the first call on each device and cached with the id of
// the CUDA context it belongs to. A later call in another context of that device (after
// cudaDeviceReset) looks it up again; a call whose context id cannot be read looks it up every
// time.
int noalloc_scratch(tpmlp_ctx* c, void** out) {
    if (c->device < 0 || c->device >= kNoallocMaxDevices) return TPMLP_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoallocSlot& slot = g_noalloc[c->device];
    unsigned long long id = current_context_id();
    if (!slot.ptr || id == 0 || id != slot.ctx_id) {
        void* p = nullptr;
        TPMLP_CUDA(c, cudaGetSymbolAddress(&p, g_noalloc_y));
        if (!p) {
            c->last_error = "cudaGetSymbolAddress returned a null scratch address";
            return TPMLP_ERR_CUDA;
        }
        if (id == 0) id = current_context_id();  // the lookup made the primary context current
        slot.ptr = p;
        slot.ctx_id = id;
    }
    *out = slot.ptr;
    return TPMLP_OK;
}

}  // namespace

extern "C" int tpmlp_forward_noalloc(tpmlp_ctx* c, const void* X, int64_t B, int64_t S, void* Z,
                                     void* stream) {
    int rc = check_ctx(c);
    if (rc) return rc;
    if ((rc = check_tokens(B, S))) return rc;
    const int64_t M = B * S;
    if (M == 0) return TPMLP_OK;
    if (!X || !Z) return TPMLP_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Z)) return TPMLP_ERR_MISALIGNED;
    const int64_t y_bytes = M * c->F * 2;
    if (y_bytes > static_cast<int64_t>(TPMLP_NOALLOC_SCRATCH_BYTES)) {
        c->last_error = "tpmlp_forward_noalloc: Y needs " + std::to_string(y_bytes) +
                        " bytes (B*S*F*2) but the static scratch holds " +
                        std::to_string(static_cast<int64_t>(TPMLP_NOALLOC_SCRATCH_BYTES)) +
                        "; use tpmlp_forward or fewer tokens per call";
        return TPMLP_ERR_UNSUPPORTED_SHAPE;
    }
    void* y = nullptr;
    if ((rc = noalloc_scratch(c, &y))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((rc = run_gemm1(c, X, M, y, s))) return rc;
    return run_gemm2(c, y, M, Z, s);
}
