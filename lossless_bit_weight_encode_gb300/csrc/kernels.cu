// Host launchers of the W12 kernels and the per-device status word.
//
// One translation unit holds every kernel so that the status word
// (g_w12_status, static device memory: no allocation) is one symbol per device.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <utility>

#include "decode.cuh"
#include "encode_gpu.cuh"
#include "gemm_tc.cuh"
#include "gemm_tc_sm.cuh"
#include "gemv.cuh"
#include "gemv_sm.cuh"
#include "w12_host.hpp"
#include "w12_launch.hpp"

namespace w12 {
namespace dev {

__device__ uint32_t g_w12_status;

// Copies x [M][K] into a zero-padded [M][K8] buffer whose rows are 16-byte
// aligned, for the tensor map (used only when x itself is not so aligned).
__global__ void w12_pad_x_kernel(const uint16_t *__restrict__ x, uint16_t *__restrict__ xp, int M, int64_t K,
                                 int64_t K8) {
    const int64_t total = (int64_t)M * K8;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / K8, k = i % K8;
        xp[i] = k < K ? x[m * K + k] : (uint16_t)0;
    }
}

// Turns the argmax keys of the LM-head GEMM back into (row index, fp32 logit).
__global__ void w12_argmax_finalize_kernel(const unsigned long long *__restrict__ keys, int M,
                                           int32_t *__restrict__ idx, float *__restrict__ val) {
    const int m = (int)threadIdx.x;
    if (m >= M) return;
    const unsigned long long k = keys[m];
    const uint32_t ord = (uint32_t)(k >> 32);
    idx[m] = (int32_t)(0xFFFFFFFFu - (uint32_t)k);
    val[m] = __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}

// Reads n16 16-byte words once (eight loads in flight per thread, streaming
// cache hint) and folds them into one word per thread, written only if it
// equals `never`: the HBM read ceiling the GEMM kernels are measured against.
__global__ void __launch_bounds__(512, 2) w12_read_stream_kernel(const uint4 *__restrict__ p, int64_t n16,
                                                             uint32_t never, uint32_t *__restrict__ sink) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t acc = 0;
    for (; i + 7 * stride < n16; i += 8 * stride) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = __ldcs(p + i + u * stride);
#pragma unroll
        for (int u = 0; u < 8; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
    for (; i < n16; i += stride) {
        const uint4 v = __ldcs(p + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    if (acc == never) sink[0] = acc;
}

// Waits on an mbarrier that nothing arrives on, with a short deadline, and
// records the timeout: exercises the bounded-wait path without a fault.
__global__ void w12_selftest_timeout_kernel(uint32_t *status, uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, globaltimer_ns() + timeout_ns)) atomicOr(status, kStatusTimeout);
}

}  // namespace dev

namespace launch {
namespace {

constexpr int kStages = 4;
constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int status_code = W12_OK;
    std::string error;
    int device = 0;
    int sm_count = 0;
    uint32_t *status = nullptr;
    int occupancy[2][2] = {{0, 0}, {0, 0}};  // [ntok==32][a_smem]
    int q8_occupancy[2] = {0, 0};            // [ntok==32], Q8 copy kernels
    int gemv_occupancy[2] = {0, 0};          // GEMV with 1, 2 token rows
    int gemv_sm_occupancy[2] = {0, 0};       // one-CTA-per-SM GEMV with 1, 2 token rows
    int tc_sm_occupancy[2][2] = {{0, 0}, {0, 0}};  // one-CTA-per-SM tensor-core kernel, [q8][ntok==32]
};

DeviceState g_state[kMaxDevices];
std::mutex g_mu;

template <int NTOK, bool ASMEM, bool Q8 = false>
void *gemm_kernel_ptr() {
    return reinterpret_cast<void *>(&dev::w12_gemm_tc_kernel<NTOK, kStages, ASMEM, Q8>);
}
template <int NTOK, bool ASMEM, bool Q8 = false>
int gemm_smem_bytes() {
    return dev::GemmCfg<NTOK, kStages, ASMEM, Q8>::kSmemBytes;
}

int cuda_fail(cudaError_t e, const char *what, std::string *err) {
    *err = std::string(what) + ": " + cudaGetErrorString(e);
    return W12_ERR_CUDA;
}

// Resident CTAs per SM from the kernel's own limits: registers (allocated per
// warp in units of 256), dynamic shared memory (+1 KB reserved per CTA) and
// threads.  The runtime's occupancy query is taken when it reports more.
int resident_ctas(const void *kernel, int threads, int smem_bytes, int device, std::string *err, int *out) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes", err);
    int regs_sm = 0, smem_sm = 0, threads_sm = 0;
    cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, device);
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device);
    cudaDeviceGetAttribute(&threads_sm, cudaDevAttrMaxThreadsPerMultiProcessor, device);
    const int warps = (threads + 31) / 32;
    const int regs_warp = ((fa.numRegs * 32 + 255) / 256) * 256;
    int occ = regs_warp > 0 ? regs_sm / (warps * regs_warp) : 1;
    occ = std::min(occ, smem_sm / (smem_bytes + 1024));
    occ = std::min(occ, threads_sm / threads);
    int api = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&api, kernel, threads, (size_t)smem_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor", err);
    *out = std::max(std::max(occ, api), 1);
    return W12_OK;
}

template <int NTOK, bool ASMEM, bool Q8 = false>
int prepare_gemm(DeviceState &s, std::string *err) {
    void *k = gemm_kernel_ptr<NTOK, ASMEM, Q8>();
    cudaError_t e =
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, gemm_smem_bytes<NTOK, ASMEM, Q8>());
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute", err);
    // all of the unified L1/shared storage as shared memory, so that several
    // CTAs fit on an SM
    e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(carveout)", err);
    int occ = 0;
    const int rc = resident_ctas(k, dev::GemmCfg<NTOK, kStages, ASMEM, Q8>::kThreads,
                                 gemm_smem_bytes<NTOK, ASMEM, Q8>(), s.device, err, &occ);
    if (rc != W12_OK) return rc;
    // TMEM: a 16-token CTA holds 128 of the SM's 512 columns, a 32-token CTA
    // 256; no more CTAs may be resident than their columns allow
    constexpr int kTmemCap = 512 / dev::GemmCfg<NTOK, kStages, ASMEM, Q8>::kTmemCols;
    if (occ > kTmemCap) occ = kTmemCap;
    if (Q8)
        s.q8_occupancy[NTOK == 32] = occ;
    else
        s.occupancy[NTOK == 32][ASMEM] = occ;
    return W12_OK;
}

constexpr int kGemvStages = 4;
constexpr int kGemvChunks = 4;  // chunks per weight stage
template <int MT>
using GemvC = dev::GemvCfg<kGemvStages, kGemvChunks, MT>;

template <int MT>
int prepare_gemv(DeviceState &s, std::string *err) {
    void *k = reinterpret_cast<void *>(&dev::w12_gemv_kernel<kGemvStages, kGemvChunks, MT>);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, GemvC<MT>::kSmemBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(gemv)", err);
    e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(gemv carveout)", err);
    int occ = 0;
    const int rc = resident_ctas(k, GemvC<MT>::kThreads, GemvC<MT>::kSmemBytes, s.device, err, &occ);
    if (rc != W12_OK) return rc;
    s.gemv_occupancy[MT - 1] = occ < 8 ? occ : 8;
    return W12_OK;
}

template <int MT>
int prepare_gemv_sm(DeviceState &s, std::string *err) {
    using C = dev::GemvSmCfg<MT>;
    void *k = reinterpret_cast<void *>(&dev::w12_gemv_sm_kernel<MT>);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(gemv_sm)", err);
    e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(gemv_sm carveout)", err);
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, C::kThreads, (size_t)C::kSmemBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(gemv_sm)", err);
    s.gemv_sm_occupancy[MT - 1] = occ;
    return W12_OK;
}

template <int NTOK, bool Q8>
int prepare_tc_sm(DeviceState &s, std::string *err) {
    using C = dev::TcSmCfg<NTOK, Q8>;
    void *k = reinterpret_cast<void *>(&dev::w12_gemm_tc_sm_kernel<NTOK, Q8>);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(tc_sm)", err);
    e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(tc_sm carveout)", err);
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, C::kThreads, (size_t)C::kSmemBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(tc_sm)", err);
    // all 512 TMEM columns: one CTA per SM whatever else would fit
    s.tc_sm_occupancy[Q8][NTOK == 32] = occ < 1 ? occ : 1;
    return W12_OK;
}

// Per-device set-up on first use (with that device current).
int device_state(DeviceState **out, std::string *err) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice", err);
    if (dev < 0 || dev >= kMaxDevices) {
        *err = "device ordinal out of range";
        return W12_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &s = g_state[dev];
    if (!s.ready) {
        s.device = dev;
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        e = cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute", err);
        if (major != 10 || minor != 3) {
            *err = "W12 kernels are built for sm_103a (compute capability 10.3); this device is " +
                   std::to_string(major) + "." + std::to_string(minor);
            return W12_ERR_UNSUPPORTED_ARCH;
        }
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&s.status), dev::g_w12_status);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)", err);
        int rc = prepare_gemv<1>(s, err);
        if (rc == W12_OK) rc = prepare_gemv<2>(s, err);
        if (rc == W12_OK) rc = prepare_gemv_sm<1>(s, err);
        if (rc == W12_OK) rc = prepare_gemv_sm<2>(s, err);
        if (rc == W12_OK) rc = prepare_gemm<16, false>(s, err);
        if (rc == W12_OK) rc = prepare_gemm<32, false>(s, err);
        if (rc == W12_OK) rc = prepare_gemm<16, true>(s, err);
        if (rc == W12_OK) rc = prepare_gemm<32, true>(s, err);
        if (rc == W12_OK) rc = prepare_tc_sm<16, false>(s, err);
        if (rc == W12_OK) rc = prepare_tc_sm<32, false>(s, err);
        if (rc == W12_OK) rc = prepare_tc_sm<16, true>(s, err);
        if (rc == W12_OK) rc = prepare_tc_sm<32, true>(s, err);
        if (rc == W12_OK) rc = prepare_gemm<16, false, true>(s, err);
        if (rc == W12_OK) rc = prepare_gemm<32, false, true>(s, err);
        if (rc != W12_OK) return rc;
        s.ready = true;
    }
    *out = &s;
    return W12_OK;
}

// Launch options (w12_set_option).  Process-wide, read with relaxed atomics
// on every call; nothing is taken from the environment.
struct OptionSlot {
    const char *name;
    int64_t def, lo, hi;
    std::atomic<int64_t> value;
};

// name, default, smallest and largest accepted value
OptionSlot g_options[] = {
    // largest M on the CUDA-core path (0: every M on the tensor cores); four
    // token rows on CUDA cores measured 35 % slower than tcgen05
    {"gemv_max_m", 2, 0, 2, {2}},
    // token tile of the tensor-core kernel: 0 picks (see tc_token_tile)
    {"token_tile", 0, 0, 32, {0}},
    // 1: the tensor-core kernel takes its A operand from shared memory
    {"a_operand_smem", 0, 0, 1, {0}},
    // CUDA-core kernel: -1 picks, 0 two CTAs per SM, 1 one CTA per SM
    {"gemv_sm", -1, -1, 1, {-1}},
    // 0: fixed split-K for the CUDA-core kernel too (no stream-K ranges)
    {"stream_k", 1, 0, 1, {1}},
    // 0: the planner picks; n: fixed split-K with n splits where it fits
    {"splits", 0, 0, 1 << 20, {0}},
    // 0: launches without programmatic dependent launch
    {"pdl", 1, 0, 1, {1}},
    // bounded waits give up after this many milliseconds
    {"timeout_ms", 4000, 1, 600000, {4000}},
    // tensor-core path: 1 one CTA per SM (stream-K ranges), 0 several CTAs per
    // SM with fixed split-K
    {"tc_sm", 1, 0, 1, {1}},
};

enum OptionId {
    kOptGemvMaxM,
    kOptTokenTile,
    kOptASmem,
    kOptGemvSm,
    kOptStreamK,
    kOptSplits,
    kOptPdl,
    kOptTimeout,
    kOptTcSm
};

int64_t opt(OptionId id) { return g_options[id].value.load(std::memory_order_relaxed); }

// One and two tokens run on CUDA cores unless gemv_max_m says fewer.
bool use_gemv(int M) { return M <= 2 && M <= opt(kOptGemvMaxM); }

// Token tile of the tensor-core kernel.  32 unless the matrix has enough
// 128-row tiles for several waves (a 152K-row LM head): two CTAs per SM with
// the 32-token tile measured 160 us per grouped layer step at M = 4..16
// against 190 us for three CTAs per SM with the 16-token tile, while the LM
// head took 268 us with the 16-token tile against 303 us.  token_tile = 16 or
// 32 forces one (kept tested); more than 16 tokens always take 32.
int tc_token_tile(int M, int64_t tiles, int sm_count) {
    const int64_t v = opt(kOptTokenTile);
    if (v == 32 || M > 16) return 32;
    if (v == 16) return 16;
    return tiles >= 3 * (int64_t)sm_count ? 16 : 32;
}

bool use_smem_a_operand() { return opt(kOptASmem) != 0; }

// The one-CTA-per-SM tensor-core kernel (gemm_tc_sm.cuh) takes its A operand
// from TMEM only; the shared-memory A variant stays on the several-CTA kernel.
bool use_tc_sm() { return opt(kOptTcSm) != 0 && !use_smem_a_operand(); }

// Token tile of the one-CTA-per-SM tensor-core kernel: the narrowest MMA
// (N = 16) that holds M tokens, unless token_tile forces 32.
int tc_sm_token_tile(int M) { return (M > 16 || opt(kOptTokenTile) == 32) ? 32 : 16; }

// Which CUDA-core kernel: one CTA per SM with sixteen decode warps (gemv_sm.cuh)
// or two with eight each (gemv.cuh).  The first keeps every warp of an SM busy
// to the end of a single wave.  Measured (one GPU, back to back): layer step at
// M = 1 / 2 110.1 / 124.6 us against 115.7 / 134.2; the LM head 199.0 against
// 209.1 us; heavy-tail weights (0.4 % escapes, nearly every quarter-chunk
// holding some) 169.1 / 187.9 against 175.2 / 191.7 us once each warp finds
// its escapes' offset from the nearer end of its quarter.  So one CTA per SM
// whenever one wave of ranges of at most kMaxSegs segments covers the launch;
// gemv_sm = 0 or 1 forces a kernel.
bool use_gemv_sm(const w12_info &info, int sm_count) {
    const int64_t v = opt(kOptGemvSm);
    if (v >= 0) return v == 1;
    const int64_t units = info.tiles * info.segs;
    return (units + sm_count - 1) / sm_count <= dev::GemvSmCfg<1>::kMaxSegs;
}

// The GEMV shares a single wave's work as stream-K unit ranges unless
// stream_k = 0 (then fixed split-K as for the tensor-core kernel).
bool use_stream_k() { return opt(kOptStreamK) != 0; }

uint64_t timeout_ns() { return (uint64_t)opt(kOptTimeout) * 1000000ull; }

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder(std::string *err) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    if (!fn) *err = "cuTensorMapEncodeTiled is not available from the driver";
    return fn;
}

}  // namespace

int plan_gemm(const w12_info &info, int M, GemmPlan *plan, std::string *err, bool q8) {
    if (M < 1 || M > 32) {
        *err = "M must be in 1..32";
        return W12_ERR_INVALID_ARG;
    }
    DeviceState *s = nullptr;
    int rc = device_state(&s, err);
    if (rc != W12_OK) return rc;
    plan->gemv = !q8 && use_gemv(M);
    plan->gemv_sm = plan->gemv && use_gemv_sm(info, s->sm_count);
    plan->tc_sm = !plan->gemv && use_tc_sm();
    plan->ntok = plan->gemv ? M : plan->tc_sm ? tc_sm_token_tile(M) : tc_token_tile(M, info.tiles, s->sm_count);
    const int occ = plan->gemv_sm ? s->gemv_sm_occupancy[M - 1]
                    : plan->gemv  ? s->gemv_occupancy[M - 1]
                    : plan->tc_sm ? s->tc_sm_occupancy[q8][plan->ntok == 32]
                    : q8          ? s->q8_occupancy[plan->ntok == 32]
                                  : s->occupancy[plan->ntok == 32][use_smem_a_operand()];
    if (occ < 1) {
        *err = "GEMM kernel cannot be resident on this device";
        return W12_ERR_CUDA;
    }
    const int64_t kMaxSegs = plan->gemv_sm ? dev::GemvSmCfg<1>::kMaxSegs
                             : plan->tc_sm ? dev::TcSmCfg<16>::kMaxSegs
                                           : dev::GemmCfg<16, kStages, false>::kMaxSegs;
    static_assert(dev::TcSmCfg<16>::kMaxSegs == dev::TcSmCfg<32>::kMaxSegs &&
                      dev::TcSmCfg<16>::kMaxPieces == dev::TcSmCfg<32>::kMaxPieces,
                  "one range limit for both token tiles");
    const int64_t capacity = (int64_t)s->sm_count * occ;
    const int64_t tiles = info.tiles, segs = info.segs;
    const int64_t forced = opt(kOptSplits);  // tuning override: fixed split-K
    plan->units = 0;
    // one wave of equal contiguous unit ranges (stream-K): no SM idles
    // because the tile count does not divide the resident CTA count
    const int64_t units = tiles * segs;
    int64_t sk_ctas = capacity < units ? capacity : units;
    // the one-CTA-per-SM kernels give each CTA at least kMinRange segments:
    // below that a CTA's fixed costs (first stage, split-K finish) outweigh its
    // streaming, and a small matrix (1024 x 5120: 160 segments) would split
    // every tile twenty ways
    constexpr int64_t kMinRange = 4;
    if ((plan->gemv_sm || plan->tc_sm) && units < kMinRange * sk_ctas)
        sk_ctas = std::max<int64_t>(1, units / kMinRange);
    // the range of a CTA: at most kMaxSegs segment headers and, for the
    // one-CTA-per-SM kernel, at most kMaxPieces tiles; for the two-CTA kernel
    // at most two tiles (a single wave of more CTAs than tiles)
    const int64_t max_range =
        plan->gemv_sm  ? std::min<int64_t>(kMaxSegs, (dev::GemvSmCfg<1>::kMaxPieces - 1) * segs + 1)
        : plan->tc_sm ? std::min<int64_t>(kMaxSegs, (dev::TcSmCfg<16>::kMaxPieces - 1) * segs + 1)
                      : kMaxSegs;
    if ((units + sk_ctas - 1) / sk_ctas > max_range) sk_ctas = (units + max_range - 1) / max_range;
    const bool sk_shape = plan->gemv_sm || plan->tc_sm || tiles < capacity;
    // (the device computes unit x ctas products in 32 bits)
    if ((plan->gemv || plan->tc_sm) && forced == 0 && sk_shape && units * sk_ctas < (int64_t(1) << 31) && use_stream_k()) {
        const int64_t shortest = units / sk_ctas;  // units of the shortest range
        plan->units = units;
        // most ranges one tile can meet: the one holding its first unit plus
        // at most 1 + (segs - 2) / shortest range starts inside it
        plan->splits = (int)(segs == 1 ? 1 : 2 + (segs - 2) / shortest);
        plan->ctas = (int)sk_ctas;
    } else {
        int64_t splits = capacity / tiles;
        if (splits < 1) splits = 1;
        if (splits > segs) splits = segs;
        int64_t per = (segs + splits - 1) / splits;          // segments of the longest CTA
        if (per > kMaxSegs) per = kMaxSegs;
        splits = (segs + per - 1) / per;                      // fewest splits with that length
        if (forced != 0 && forced <= segs && (segs + forced - 1) / forced <= kMaxSegs) splits = forced;
        plan->splits = (int)splits;
        plan->ctas = (int)(tiles * splits);
    }
    const int64_t splits = plan->splits;
    plan->ctas_per_sm = occ;
    plan->kernel = plan->gemv_sm ? W12_KERNEL_GEMV_SM
                   : plan->gemv  ? W12_KERNEL_GEMV
                   : plan->tc_sm ? W12_KERNEL_TC_SM
                                 : W12_KERNEL_TC;
    const int64_t k8 = (info.K + 7) / 8 * 8;
    plan->ws_counters = 0;
    plan->ws_partials = up256((size_t)tiles * 4);
    const size_t partial_bytes = splits > 1 ? up256((size_t)splits * (size_t)M * (size_t)info.N_pad * 4) : 0;
    plan->ws_x = plan->ws_partials + partial_bytes;
    plan->ws_bytes = plan->ws_x + up256((size_t)M * (size_t)k8 * 2);
    return W12_OK;
}

int read_stream(const void *buf_dev, size_t bytes, void *sink_dev, uint32_t never, void *stream, std::string *err) {
    DeviceState *s = nullptr;
    int rc = device_state(&s, err);
    if (rc != W12_OK) return rc;
    // two resident CTAs of 512 threads per SM (64 registers each), eight
    // 16-byte loads in flight per thread: 128 KB per SM
    const int64_t n16 = (int64_t)(bytes / 16);
    const unsigned grid = (unsigned)(2 * s->sm_count);
    dev::w12_read_stream_kernel<<<grid, 512, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(buf_dev), n16, never, static_cast<uint32_t *>(sink_dev));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "read-stream launch", err);
    return W12_OK;
}

int decode(const void *blob_dev, const w12_info &info, uint16_t *out_dev, void *stream, std::string *err) {
    DeviceState *s = nullptr;
    int rc = device_state(&s, err);
    if (rc != W12_OK) return rc;
    dev::DecodeParams p;
    p.blob = static_cast<const uint8_t *>(blob_dev);
    p.off_seg = info.off_seghdr;
    p.off_w = info.off_weights;
    p.off_esc = info.off_escapes;
    p.N = info.N;
    p.K = info.K;
    p.chunks = info.chunks;
    p.segs = info.segs;
    p.out = out_dev;
    dim3 grid((unsigned)info.segs, (unsigned)info.tiles);
    dev::w12_decode_kernel<<<grid, 128, 0, static_cast<cudaStream_t>(stream)>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "decode launch", err);
    return W12_OK;
}

namespace {
// GEMM launches carry the programmatic-stream-serialization attribute: the
// kernel may start while the previous kernel in the stream finishes; it warms
// L2 with its first weights and then waits (griddepcontrol.wait) before any
// other memory access.  The option pdl = 0 turns the attribute off.
bool use_pdl() { return opt(kOptPdl) != 0; }

template <class... KArgs, class... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = use_pdl() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <int NTOK, bool ASMEM, bool Q8 = false>
cudaError_t launch_gemm_kernel(const dev::GemmGroup &p, const CUtensorMap &tm, int splits, int64_t tiles,
                               cudaStream_t st) {
    dim3 grid((unsigned)splits, (unsigned)tiles);
    return launch_overlapped(dev::w12_gemm_tc_kernel<NTOK, kStages, ASMEM, Q8>, grid,
                             dim3(dev::GemmCfg<NTOK, kStages, ASMEM, Q8>::kThreads),
                             (size_t)gemm_smem_bytes<NTOK, ASMEM, Q8>(), st, p, tm);
}
}  // namespace

namespace {
int gemm_impl(const uint16_t *x_dev, int count, const void *const *blobs, const w12_info *infos,
              uint16_t *const *ys, unsigned long long *amax, int M, void *workspace, size_t ws_bytes, void *stream,
              std::string *err, const w12_q8_info *q8 = nullptr);  // q8: one info per matrix, or null
int gemm_impl(const uint16_t *x_dev, const void *blob_dev, const w12_info &info, uint16_t *y_dev,
              unsigned long long *amax, int M, void *workspace, size_t ws_bytes, void *stream, std::string *err,
              const w12_q8_info *q8 = nullptr) {
    uint16_t *ys[1] = {y_dev};
    return gemm_impl(x_dev, 1, &blob_dev, &info, ys, amax, M, workspace, ws_bytes, stream, err, q8);
}

// The matrices of a group share x, so K; they are planned as one matrix of all
// their tiles (one split count) and each gets its own share of the workspace.
w12_info group_info(int count, const w12_info *infos) {
    w12_info g = infos[0];
    for (int i = 1; i < count; ++i) {
        g.tiles += infos[i].tiles;
        g.N_pad += infos[i].N_pad;
        g.N += infos[i].N;
        g.n_escapes += infos[i].n_escapes;
    }
    return g;
}

// The planner and launcher work on a w12_info; a Q8 copy has the same grid.
w12_info q8_as_info(const w12_q8_info &q) {
    w12_info i{};
    i.N = q.N;
    i.K = q.K;
    i.N_pad = q.N_pad;
    i.K_pad = q.K_pad;
    i.tiles = q.tiles;
    i.chunks = q.chunks;
    i.segs = q.segs;
    i.off_weights = q.off_q;
    i.total_bytes = q.total_bytes;
    return i;
}
}  // namespace

int q8_workspace_size(const w12_q8_info &info, int M, size_t *bytes, std::string *err) {
    GemmPlan plan;
    const int rc = plan_gemm(q8_as_info(info), M, &plan, err, true);
    if (rc == W12_OK) *bytes = plan.ws_bytes;
    return rc;
}

int q8_gemm(const uint16_t *x_dev, const void *blob_dev, const w12_q8_info &info, uint16_t *y_dev, int M,
            void *workspace, size_t ws_bytes, void *stream, std::string *err) {
    return gemm_impl(x_dev, blob_dev, q8_as_info(info), y_dev, nullptr, M, workspace, ws_bytes, stream, err, &info);
}

namespace {
// The w12_info views of a Q8 group (count <= kMaxGroup, checked by the caller).
void q8_group_infos(int count, const w12_q8_info *q8, w12_info (&infos)[dev::kMaxGroup]) {
    for (int i = 0; i < count; ++i) infos[i] = q8_as_info(q8[i]);
}
}  // namespace

int q8_group_plan(int count, const w12_q8_info *q8, int M, GemmPlan *plan, std::string *err) {
    w12_info infos[dev::kMaxGroup];
    q8_group_infos(count, q8, infos);
    return plan_gemm(group_info(count, infos), M, plan, err, true);
}

int q8_group_workspace_size(int count, const w12_q8_info *q8, int M, size_t *bytes, std::string *err) {
    GemmPlan plan;
    const int rc = q8_group_plan(count, q8, M, &plan, err);
    if (rc == W12_OK) *bytes = plan.ws_bytes;
    return rc;
}

int q8_gemm_group(const uint16_t *x_dev, int count, const void *const *blobs, const w12_q8_info *q8,
                  uint16_t *const *ys, int M, void *workspace, size_t ws_bytes, void *stream, std::string *err) {
    w12_info infos[dev::kMaxGroup];
    q8_group_infos(count, q8, infos);
    return gemm_impl(x_dev, count, blobs, infos, ys, nullptr, M, workspace, ws_bytes, stream, err, q8);
}

int gemm(const uint16_t *x_dev, const void *blob_dev, const w12_info &info, uint16_t *y_dev, int M,
         void *workspace, size_t ws_bytes, void *stream, std::string *err) {
    return gemm_impl(x_dev, blob_dev, info, y_dev, nullptr, M, workspace, ws_bytes, stream, err);
}

int group_plan(int count, const w12_info *infos, int M, GemmPlan *plan, std::string *err) {
    return plan_gemm(group_info(count, infos), M, plan, err);
}

int group_workspace_size(int count, const w12_info *infos, int M, size_t *bytes, std::string *err) {
    GemmPlan plan;
    const int rc = plan_gemm(group_info(count, infos), M, &plan, err);
    if (rc == W12_OK) *bytes = plan.ws_bytes;
    return rc;
}

int gemm_group(const uint16_t *x_dev, int count, const void *const *blobs, const w12_info *infos,
               uint16_t *const *ys, int M, void *workspace, size_t ws_bytes, void *stream, std::string *err) {
    return gemm_impl(x_dev, count, blobs, infos, ys, nullptr, M, workspace, ws_bytes, stream, err);
}

int argmax_workspace_size(const w12_info &info, int M, size_t *bytes, std::string *err) {
    GemmPlan plan;
    const int rc = plan_gemm(info, M, &plan, err);
    if (rc != W12_OK) return rc;
    *bytes = up256(plan.ws_bytes) + up256(sizeof(unsigned long long) * (size_t)M);
    return W12_OK;
}

int gemm_argmax(const uint16_t *x_dev, const void *blob_dev, const w12_info &info, int M, uint16_t *y_dev,
                int32_t *idx_dev, float *val_dev, void *workspace, size_t ws_bytes, void *stream, std::string *err) {
    GemmPlan plan;
    int rc = plan_gemm(info, M, &plan, err);
    if (rc != W12_OK) return rc;
    const size_t keys_off = up256(plan.ws_bytes);
    if (ws_bytes < keys_off + up256(sizeof(unsigned long long) * (size_t)M)) {
        *err = "workspace smaller than w12_gemm_argmax_workspace_size";
        return W12_ERR_BUFFER_TOO_SMALL;
    }
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto *keys = reinterpret_cast<unsigned long long *>(static_cast<uint8_t *>(workspace) + keys_off);
    cudaError_t e = cudaMemsetAsync(keys, 0, sizeof(unsigned long long) * (size_t)M, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(argmax keys)", err);
    rc = gemm_impl(x_dev, blob_dev, info, y_dev, keys, M, workspace, keys_off, stream, err);
    if (rc != W12_OK) return rc;
    dev::w12_argmax_finalize_kernel<<<1, 32, 0, st>>>(keys, M, idx_dev, val_dev);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "argmax finalize launch", err);
    return W12_OK;
}

namespace {
int gemm_impl(const uint16_t *x_dev, int count, const void *const *blobs, const w12_info *infos,
              uint16_t *const *ys, unsigned long long *amax, int M, void *workspace, size_t ws_bytes, void *stream,
              std::string *err, const w12_q8_info *q8) {
    const w12_info info = group_info(count, infos);
    GemmPlan plan;
    int rc = plan_gemm(info, M, &plan, err, q8 != nullptr);
    if (rc != W12_OK) return rc;
    if (ws_bytes < plan.ws_bytes) {
        *err = "workspace smaller than w12_gemm_workspace_size";
        return W12_ERR_BUFFER_TOO_SMALL;
    }
    DeviceState *s = nullptr;
    rc = device_state(&s, err);
    if (rc != W12_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);

    // x must be a TMA source: 16-byte aligned rows (K % 8 == 0, aligned base)
    const uint16_t *xsrc = x_dev;
    int64_t ld = info.K;
    if ((reinterpret_cast<uintptr_t>(x_dev) & 15) != 0 || (info.K & 7) != 0) {
        ld = (info.K + 7) / 8 * 8;
        uint16_t *xp = reinterpret_cast<uint16_t *>(ws + plan.ws_x);
        const int64_t total = (int64_t)M * ld;
        const int blocks = (int)((total + 255) / 256 < 1024 ? (total + 255) / 256 : 1024);
        dev::w12_pad_x_kernel<<<blocks, 256, 0, st>>>(x_dev, xp, M, info.K, ld);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "x padding launch", err);
        xsrc = xp;
    }
    auto encode = tensor_map_encoder(err);
    if (!encode) return W12_ERR_CUDA;
    CUtensorMap tm;
    const cuuint64_t dims[2] = {(cuuint64_t)info.K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    // tensor cores: 64-column boxes of NTOK token rows, 128-byte swizzle;
    // GEMV: one 256-column box of the single row, no swizzle
    const cuuint32_t box[2] = {plan.gemv ? (cuuint32_t)kSegK : 64u, (cuuint32_t)plan.ntok};
    const cuuint32_t estr[2] = {1u, 1u};
    CUresult cr = encode(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(xsrc), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         plan.gemv ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed for x (code " + std::to_string((int)cr) + ")";
        return W12_ERR_CUDA;
    }

    dev::GemmGroup p{};
    p.n = count;
    p.units = (int32_t)plan.units;
    p.ctas = plan.ctas;
    int64_t tile0 = 0, npad0 = 0;
    for (int i = 0; i < count; ++i) {
        const w12_info &mi = infos[i];
        dev::GemmParams &q = p.m[i];
        q.blob = static_cast<const uint8_t *>(blobs[i]);
        q.off_seg = mi.off_seghdr;
        q.off_w = mi.off_weights;
        q.off_esc = mi.off_escapes;
        q.N = mi.N;
        q.Npad = mi.N_pad;
        q.chunks = (int32_t)mi.chunks;
        q.segs = (int32_t)mi.segs;
        q.M = M;
        q.splits = plan.splits;
        q.partials = reinterpret_cast<float *>(ws + plan.ws_partials) + (size_t)plan.splits * (size_t)M * (size_t)npad0;
        q.counters = reinterpret_cast<uint32_t *>(ws + plan.ws_counters) + tile0;
        q.y = ys[i];
        q.amax = amax;
        q.scales = q8 ? reinterpret_cast<const float *>(q.blob + q8[i].off_scales) : nullptr;
        q.status = s->status;
        q.timeout_ns = timeout_ns();
        p.tile0[i] = tile0;
        tile0 += mi.tiles;
        npad0 += mi.N_pad;
    }
    for (int i = count; i <= dev::kMaxGroup; ++i) p.tile0[i] = tile0;

    cudaError_t e;
    const bool asmem = use_smem_a_operand();
    if (plan.gemv) {
        const dim3 grid = plan.units > 0 ? dim3((unsigned)plan.ctas, 1u) : dim3((unsigned)plan.splits, (unsigned)info.tiles);
        if (plan.gemv_sm && plan.ntok == 1)
            e = launch_overlapped(dev::w12_gemv_sm_kernel<1>, grid, dim3(dev::GemvSmCfg<1>::kThreads),
                                  (size_t)dev::GemvSmCfg<1>::kSmemBytes, st, p, tm);
        else if (plan.gemv_sm)
            e = launch_overlapped(dev::w12_gemv_sm_kernel<2>, grid, dim3(dev::GemvSmCfg<2>::kThreads),
                                  (size_t)dev::GemvSmCfg<2>::kSmemBytes, st, p, tm);
        else if (plan.ntok == 1)
            e = launch_overlapped(dev::w12_gemv_kernel<kGemvStages, kGemvChunks, 1>, grid, dim3(GemvC<1>::kThreads),
                                  (size_t)GemvC<1>::kSmemBytes, st, p, tm);
        else
            e = launch_overlapped(dev::w12_gemv_kernel<kGemvStages, kGemvChunks, 2>, grid, dim3(GemvC<2>::kThreads),
                                  (size_t)GemvC<2>::kSmemBytes, st, p, tm);
    } else if (plan.tc_sm) {
        const dim3 grid = plan.units > 0 ? dim3((unsigned)plan.ctas, 1u) : dim3((unsigned)plan.splits, (unsigned)info.tiles);
        if (q8 && plan.ntok == 16)
            e = launch_overlapped(dev::w12_gemm_tc_sm_kernel<16, true>, grid, dim3(dev::TcSmCfg<16, true>::kThreads),
                                  (size_t)dev::TcSmCfg<16, true>::kSmemBytes, st, p, tm);
        else if (q8)
            e = launch_overlapped(dev::w12_gemm_tc_sm_kernel<32, true>, grid, dim3(dev::TcSmCfg<32, true>::kThreads),
                                  (size_t)dev::TcSmCfg<32, true>::kSmemBytes, st, p, tm);
        else if (plan.ntok == 16)
            e = launch_overlapped(dev::w12_gemm_tc_sm_kernel<16>, grid, dim3(dev::TcSmCfg<16>::kThreads),
                                  (size_t)dev::TcSmCfg<16>::kSmemBytes, st, p, tm);
        else
            e = launch_overlapped(dev::w12_gemm_tc_sm_kernel<32>, grid, dim3(dev::TcSmCfg<32>::kThreads),
                                  (size_t)dev::TcSmCfg<32>::kSmemBytes, st, p, tm);
    } else if (q8) {
        e = plan.ntok == 16 ? launch_gemm_kernel<16, false, true>(p, tm, plan.splits, info.tiles, st)
                            : launch_gemm_kernel<32, false, true>(p, tm, plan.splits, info.tiles, st);
    } else if (plan.ntok == 16)
        e = asmem ? launch_gemm_kernel<16, true>(p, tm, plan.splits, info.tiles, st)
                  : launch_gemm_kernel<16, false>(p, tm, plan.splits, info.tiles, st);
    else
        e = asmem ? launch_gemm_kernel<32, true>(p, tm, plan.splits, info.tiles, st)
                  : launch_gemm_kernel<32, false>(p, tm, plan.splits, info.tiles, st);
    if (e != cudaSuccess) return cuda_fail(e, "gemm launch", err);
    return W12_OK;
}
}  // namespace

int check_status(void *stream, std::string *err) {
    DeviceState *s = nullptr;
    int rc = device_state(&s, err);
    if (rc != W12_OK) return rc;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize", err);
    uint32_t v = 0;
    e = cudaMemcpy(&v, s->status, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the status word", err);
    if (v != 0) {
        const uint32_t zero = 0;
        cudaMemcpy(s->status, &zero, sizeof zero, cudaMemcpyHostToDevice);
        const std::string word = " (status word " + std::to_string(v) + ")";
        if (v & dev::kStatusTimeout) {
            *err = "a W12 kernel gave up a bounded wait" + word;
            return W12_ERR_TIMEOUT;
        }
        if (v & dev::kStatusEncodeOverflow) {
            *err = "w12_encode_device: the blob buffer is shorter than the encoding" + word;
            return W12_ERR_BUFFER_TOO_SMALL;
        }
        *err = "w12_encode_device: more than 2^32-1 escapes, split the matrix" + word;
        return W12_ERR_SHAPE;
    }
    return W12_OK;
}

// ---------------------------------------------------------------- encoder
namespace {

struct EncodeLayout {
    size_t plan = 0, base = 0, n_esc = 0, bytes = 0;
};

EncodeLayout encode_layout(const Geometry &g) {
    const size_t nseg = (size_t)(g.tiles * g.segs);
    EncodeLayout l;
    l.plan = 0;
    l.base = up256(nseg * 32);
    l.n_esc = l.base + up256(nseg * sizeof(uint64_t));
    l.bytes = l.n_esc + 256;
    return l;
}

int encode_launch(const uint16_t *w_dev, int64_t N, int64_t K, uint8_t *blob_dev, size_t cap, void *workspace,
                  size_t ws_bytes, bool write, void *stream, std::string *err) {
    if (!host::check_shape(N, K, err)) return W12_ERR_SHAPE;
    DeviceState *s = nullptr;
    int rc = device_state(&s, err);
    if (rc != W12_OK) return rc;
    const Geometry g = Geometry::of(N, K);
    const EncodeLayout l = encode_layout(g);
    if (ws_bytes < l.bytes) {
        *err = "encoder workspace smaller than w12_encode_workspace_size";
        return W12_ERR_BUFFER_TOO_SMALL;
    }
    if (write && cap < g.off_esc) {
        *err = "blob buffer smaller than the encoded size";
        return W12_ERR_BUFFER_TOO_SMALL;
    }
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    dev::EncodeParams p;
    p.w = w_dev;
    p.N = g.N;
    p.K = g.K;
    p.Kp = g.Kpad;
    p.tiles = g.tiles;
    p.chunks = g.chunks;
    p.segs = g.segs;
    p.vec = ((reinterpret_cast<uintptr_t>(w_dev) & 15) == 0 && K % 8 == 0) ? 1 : 0;
    p.plan = ws + l.plan;
    p.base = reinterpret_cast<uint64_t *>(ws + l.base);
    p.n_esc = reinterpret_cast<uint64_t *>(ws + l.n_esc);
    p.blob = blob_dev;
    p.blob_bytes = cap;
    p.off_seg = g.off_seg;
    p.off_w = g.off_w;
    p.off_esc = g.off_esc;
    p.status = s->status;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t nseg = g.tiles * g.segs;
    // plan: 34 KB of shared memory per CTA, several CTAs per SM
    const int grid = (int)std::min<int64_t>(nseg, (int64_t)s->sm_count * 6);
    dev::w12_encode_plan_kernel<<<grid, 256, 0, st>>>(p);
    dev::w12_encode_scan_kernel<<<1, 1024, 0, st>>>(p);
    if (write) {
        const int wgrid = (int)std::min<int64_t>(nseg, (int64_t)s->sm_count * 16);
        dev::w12_encode_write_kernel<<<wgrid, 128, 0, st>>>(p);
        dev::w12_encode_header_kernel<<<1, 256, 0, st>>>(p);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "encoder launch", err);
    return W12_OK;
}

}  // namespace

int encode_workspace_size(int64_t N, int64_t K, size_t *bytes, std::string *err) {
    if (!host::check_shape(N, K, err)) return W12_ERR_SHAPE;
    *bytes = encode_layout(Geometry::of(N, K)).bytes;
    return W12_OK;
}

int encoded_size_device(const uint16_t *w_dev, int64_t N, int64_t K, void *workspace, size_t ws_bytes,
                        size_t *bytes, void *stream, std::string *err) {
    int rc = encode_launch(w_dev, N, K, nullptr, 0, workspace, ws_bytes, false, stream, err);
    if (rc != W12_OK) return rc;
    const Geometry g = Geometry::of(N, K);
    const EncodeLayout l = encode_layout(g);
    uint64_t n_esc = 0;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&n_esc, static_cast<uint8_t *>(workspace) + l.n_esc, sizeof n_esc,
                                    cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return cuda_fail(e, "reading the escape count", err);
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize", err);
    if (n_esc > 0xFFFFFFFFull) {
        *err = "more than 2^32-1 escapes: split the matrix";
        return W12_ERR_SHAPE;
    }
    *bytes = (size_t)g.total(n_esc);
    return W12_OK;
}

int encode_device(const uint16_t *w_dev, int64_t N, int64_t K, void *blob_dev, size_t cap, void *workspace,
                  size_t ws_bytes, void *stream, std::string *err) {
    return encode_launch(w_dev, N, K, static_cast<uint8_t *>(blob_dev), cap, workspace, ws_bytes, true, stream,
                         err);
}

// ---------------------------------------------------------------- no-alloc
// Scratch for w12_gemm_noalloc: a fixed array in static device memory, so
// that call never allocates.  Every device that loads the library holds it
// until the process exits.  All calls share it and it keeps the last call's
// contents, so calls that overlap on the GPU race.
static __device__ __align__(256) uint8_t g_w12_noalloc_scratch[W12_NOALLOC_SCRATCH_BYTES];

namespace {
uint8_t *g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device, looked up once
// per device (with that device current): in host code the array's name is
// only a host-side stand-in, never a device address.
int noalloc_scratch(uint8_t **out, std::string *err) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice", err);
    if (dev < 0 || dev >= kMaxDevices) {
        *err = "device ordinal out of range";
        return W12_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_w12_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)", err);
        g_noalloc_ptr[dev] = static_cast<uint8_t *>(ptr);
    }
    *out = g_noalloc_ptr[dev];
    return W12_OK;
}
}  // namespace

int gemm_noalloc(const uint16_t *x_dev, const void *blob_dev, const w12_info &info, uint16_t *y_dev, int M,
                 void *stream, std::string *err) {
    GemmPlan plan;
    int rc = plan_gemm(info, M, &plan, err);
    if (rc != W12_OK) return rc;
    if (plan.ws_bytes > (size_t)W12_NOALLOC_SCRATCH_BYTES) {
        *err = "w12_gemm_noalloc: this matrix and M need " + std::to_string(plan.ws_bytes) +
               " bytes of scratch, more than the fixed " + std::to_string((size_t)W12_NOALLOC_SCRATCH_BYTES) +
               " bytes the library reserves; use w12_gemm with a caller-provided workspace";
        return W12_ERR_BUFFER_TOO_SMALL;
    }
    uint8_t *scratch = nullptr;
    rc = noalloc_scratch(&scratch, err);
    if (rc != W12_OK) return rc;
    // the split-K arrival counters must start at zero on every call
    cudaError_t e = cudaMemsetAsync(scratch + plan.ws_counters, 0, plan.ws_partials - plan.ws_counters,
                                    static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(no-alloc counters)", err);
    return gemm(x_dev, blob_dev, info, y_dev, M, scratch, (size_t)W12_NOALLOC_SCRATCH_BYTES, stream, err);
}

int set_option(const char *name, int64_t value, std::string *err) {
    for (OptionSlot &o : g_options) {
        if (std::strcmp(o.name, name) != 0) continue;
        if (value < o.lo || value > o.hi || (&o == &g_options[kOptTokenTile] && value != 0 && value != 16 &&
                                             value != 32)) {
            *err = std::string("value out of range for option ") + name;
            return W12_ERR_INVALID_ARG;
        }
        o.value.store(value, std::memory_order_relaxed);
        return W12_OK;
    }
    *err = std::string("unknown option ") + name;
    return W12_ERR_INVALID_ARG;
}

int get_option(const char *name, int64_t *value, std::string *err) {
    for (OptionSlot &o : g_options) {
        if (std::strcmp(o.name, name) != 0) continue;
        *value = o.value.load(std::memory_order_relaxed);
        return W12_OK;
    }
    *err = std::string("unknown option ") + name;
    return W12_ERR_INVALID_ARG;
}

int selftest_timeout(uint32_t timeout_us, void *stream, std::string *err) {
    DeviceState *s = nullptr;
    int rc = device_state(&s, err);
    if (rc != W12_OK) return rc;
    dev::w12_selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        s->status, (uint64_t)timeout_us * 1000ull);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "selftest launch", err);
    return W12_OK;
}

}  // namespace launch
}  // namespace w12
