// W12 decode-GEMM on tcgen05 tensor cores (sm_103a): y = x . W^T with W
// streamed from HBM in W12 form and decoded in registers.
//
// "In a memory-bound decode, reading 12 bits instead of 16 cuts weight traffic
// by a quarter" — "SpecPilot: an agent doubled speculative decoding speed, and
// the 10.87x needs context", §The mechanisms it found; the weights are
// "decoded inside the GEMM registers" (same section) and the result is
// bit-exact in the weights ("StargazerX0/SpecPilot", §What it is).
//
// Swap-AB: a CTA computes D[128 weight rows x NTOK tokens] += A . B^T where
// A = one decoded tile of W (M = 128 of the MMA) and B = x (N = 16 or 32 of the
// MMA; tokens beyond M are zeros from the TMA's out-of-bounds fill).  Each CTA
// owns one tile and a range of whole segments along K (split-K); partial sums
// go to an fp32 workspace and the last CTA of a tile adds them in split order.
//
// Warp roles (192 threads):
//   warps 0-3  decode: warp q handles rows 32q..32q+31 (TMEM lanes of quarter
//              q); per chunk it reads 48 B per row from SMEM, decodes 32
//              weights per thread, patches escapes, stores 16 columns of BF16
//              pairs into a TMEM A slot (or SMEM A slot), and later runs the
//              epilogue;
//   warp 4     producer: one lane issues cp.async.bulk for the segment
//              headers, for every stage of 2 packed chunks (12 KB) and for each
//              segment's escape bytes, plus cp.async.bulk.tensor for the
//              stage's 64-column x tile (128-byte swizzle);
//   warp 5     allocates TMEM; one lane issues tcgen05.mma (2 per chunk) and
//              tcgen05.commit.
// Every wait is bounded (deadline from %globaltimer); on expiry the kernel
// records W12_ERR_TIMEOUT in the status word, lets in-flight copies land and
// MMAs finish, frees TMEM and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "w12_device.cuh"
#include "w12_format.hpp"

namespace w12 {
namespace dev {

constexpr uint32_t kStatusTimeout = 8u;

struct GemmParams {
    const uint8_t *blob;
    uint64_t off_seg, off_w, off_esc;
    int64_t N, Npad;
    int32_t chunks, segs;     // per tile
    int32_t M, splits;
    float *partials;          // [splits][M][Npad] fp32 (splits > 1)
    uint32_t *counters;       // [tiles] arrival counters (splits > 1)
    uint16_t *y;              // [M][N] BF16
    uint32_t *status;         // device status word
    uint64_t timeout_ns;
};

template <int NTOK, int STAGES, bool A_SMEM>
struct GemmCfg {
    static constexpr int kThreads = 192;
    static constexpr int kStages = STAGES;
    static constexpr bool kASmem = A_SMEM;
    static constexpr int kNtok = NTOK;
    static constexpr int kStageChunks = 2;
    static constexpr int kWBytes = kStageChunks * kChunkBytes;  // 12288
    static constexpr int kXBytes = NTOK * 64 * 2;               // NTOK rows x 64 columns BF16
    static constexpr int kStageBytes = kWBytes + kXBytes;       // multiple of 1024
    static constexpr int kASlots = 4;
    static constexpr int kASlotBytes = kTileRows * kChunkK * 2;  // 8 KB (SMEM A variant)
    static constexpr int kEscSlots = 2;
    static constexpr int kEscCap = 2048;
    static constexpr int kMaxSegs = 96;   // segments per CTA (K range <= 24576)
    static constexpr int kTmemCols = 128;
    static constexpr int kDCol = 0;
    static constexpr int kACol = 32;
    static constexpr int kOffStages = 0;
    static constexpr int kOffA = kOffStages + STAGES * kStageBytes;
    static constexpr int kOffEsc = kOffA + (A_SMEM ? kASlots * kASlotBytes : 0);
    static constexpr int kOffHdr = kOffEsc + kEscSlots * kEscCap;
    static constexpr int kOffBars = kOffHdr + kMaxSegs * kSegHdrBytes;
    // full[S], empty[S], afull[4], aempty[4], escfull[2], escempty[2], hdr, accum, drain,
    // epi_in (partials written), epi_out (arrival counted)
    static constexpr int kNumBars = 2 * STAGES + 2 * kASlots + 2 * kEscSlots + 5;
    static constexpr int kOffMisc = kOffBars + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 64 + 1024;  // + slack to align the base to 1024
    static_assert(kStageBytes % 1024 == 0, "x tiles must stay 1024-byte aligned for the 128-byte swizzle");
    static_assert(NTOK == 16 || NTOK == 32, "token tile is 16 or 32");
};

struct Bars {
    uint64_t *full, *empty, *afull, *aempty, *escfull, *escempty, *hdr, *accum, *drain, *epi_in, *epi_out;
};

// Wait by lane 0 with a deadline, result broadcast to the warp; on success
// every lane then observes the completed phase itself.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t deadline) {
    const uint32_t lane = threadIdx.x & 31u;
    uint32_t ok = 0;
    if (lane == 0) ok = mbar_wait(bar, parity, deadline) ? 1u : 0u;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    // The phase cannot move on before this warp arrives elsewhere, so the
    // other lanes' checks succeed at once; the bound is only a safeguard.
    for (int i = 0; ok && i < (1 << 20) && !mbar_try_wait(bar, parity); ++i) {
    }
    return ok != 0;
}

// The abort flag as lane 0 sees it, so that a warp always decides as one.
__device__ __forceinline__ bool warp_aborted(volatile uint32_t *abort_flag) {
    uint32_t a = 0;
    if ((threadIdx.x & 31u) == 0) a = *abort_flag;
    return __shfl_sync(0xFFFFFFFFu, a, 0) != 0;
}

__device__ __forceinline__ void raise_timeout(uint32_t *status, volatile uint32_t *abort_flag) {
    *abort_flag = 1u;
    atomicOr(status, kStatusTimeout);
}

__device__ __forceinline__ uint16_t bf16_bits_rn(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// ------------------------------------------------------------------ producer
template <class C>
__device__ void gemm_producer(const GemmParams &p, const CUtensorMap *tmap, uint8_t *smem, const Bars &b,
                              volatile uint32_t *abort_flag, int64_t tile, int s0, int c0, int c1,
                              uint64_t deadline) {
    const int nsegs_cta = (c1 - c0 + kChunksPerSeg - 1) / kChunksPerSeg;
    const int nchunks = c1 - c0;
    const int nstages = (nchunks + 1) / 2;
    uint8_t *hdr = smem + C::kOffHdr;
    prefetch_tmap(tmap);

    // this CTA's segment headers, one copy
    const uint32_t hbytes = (uint32_t)nsegs_cta * kSegHdrBytes;
    mbar_arrive_expect_tx(b.hdr, hbytes);
    bulk_g2s(hdr, p.blob + p.off_seg + (uint64_t)(tile * p.segs + s0) * kSegHdrBytes, hbytes, b.hdr);
    bool hdr_ready = false;
    int issued = 0, esc_issued = 0;
    bool failed = false;

    for (int st = 0; st < nstages; ++st) {
        if (*abort_flag) break;
        const int chunk = c0 + 2 * st;
        if ((chunk & (kChunksPerSeg - 1)) == 0) {
            // first stage of a segment: stage its escape bytes
            const int ls = chunk / kChunksPerSeg - s0;
            const int eslot = ls & 1;
            if (!hdr_ready) {
                if (!mbar_wait(b.hdr, 0, deadline)) { failed = true; break; }
                hdr_ready = true;
            }
            if (ls >= 2 && !mbar_wait(b.escempty + eslot, (uint32_t)((ls >> 1) - 1) & 1u, deadline)) {
                failed = true;
                break;
            }
            const uint4 meta = *reinterpret_cast<const uint4 *>(hdr + ls * kSegHdrBytes + 16);
            const uint32_t base = meta.x;
            const uint32_t total = (meta.y & 0xFFFFu) + (meta.y >> 16) + (meta.z & 0xFFFFu) + (meta.z >> 16);
            if (total > 0 && total + 30u <= (uint32_t)C::kEscCap) {
                const uint32_t src0 = base & ~15u;
                const uint32_t bytes = ((base + total + 15u) & ~15u) - src0;
                mbar_arrive_expect_tx(b.escfull + eslot, bytes);
                bulk_g2s(smem + C::kOffEsc + eslot * C::kEscCap, p.blob + p.off_esc + src0, bytes, b.escfull + eslot);
            } else {
                mbar_arrive(b.escfull + eslot);  // nothing to stage (none, or read from global)
            }
            esc_issued = ls + 1;
        }
        const int slot = st % C::kStages;
        if (st >= C::kStages &&
            !mbar_wait(b.empty + slot, (uint32_t)(st / C::kStages - 1) & 1u, deadline)) {
            failed = true;
            break;
        }
        const int nch = min(2, c1 - chunk);
        uint8_t *stage = smem + C::kOffStages + slot * C::kStageBytes;
        mbar_arrive_expect_tx(b.full + slot, (uint32_t)(nch * kChunkBytes + C::kXBytes));
        bulk_g2s(stage, p.blob + p.off_w + (uint64_t)(tile * p.chunks + chunk) * kChunkBytes,
                 (uint32_t)(nch * kChunkBytes), b.full + slot);
        tma_load_2d(stage + C::kWBytes, tmap, chunk * kChunkK, 0, b.full + slot);
        issued = st + 1;
    }
    if (failed) raise_timeout(p.status, abort_flag);
    if (*abort_flag) {
        // let every copy still in flight land before the CTA can exit
        const uint64_t drain_deadline = globaltimer_ns() + 1000000000ull;
        for (int st = max(0, issued - C::kStages); st < issued; ++st)
            mbar_wait(b.full + st % C::kStages, (uint32_t)(st / C::kStages) & 1u, drain_deadline);
        for (int ls = max(0, esc_issued - 2); ls < esc_issued; ++ls)
            mbar_wait(b.escfull + (ls & 1), (uint32_t)(ls >> 1) & 1u, drain_deadline);
        mbar_wait(b.hdr, 0, drain_deadline);
    }
}

// ------------------------------------------------------------------ MMA issuer
// A chunk of 32 columns is two MMAs of K = 16.  B (x) sits in the stage's
// 128-byte-swizzled tile: K-major, rows of 128 bytes, 8-row atoms of 1024 B;
// the MMA for columns 16u..16u+15 of the stage starts 32u bytes into it.
template <class C>
__device__ void gemm_mma(const GemmParams &p, uint8_t *smem, const Bars &b, volatile uint32_t *abort_flag,
                         uint32_t tmem_base, int nchunks, uint64_t deadline) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, C::kNtok);
    bool failed = false;
    int i = 0;
    for (; i < nchunks; ++i) {
        if (*abort_flag) break;
        const int st = i >> 1, slot = st % C::kStages;
        if ((i & 1) == 0 && !mbar_wait(b.full + slot, (uint32_t)(st / C::kStages) & 1u, deadline)) {
            failed = true;
            break;
        }
        const int aslot = i % C::kASlots;
        if (!mbar_wait(b.afull + aslot, (uint32_t)(i / C::kASlots) & 1u, deadline)) {
            failed = true;
            break;
        }
        tc_fence_after();
        const uint32_t xs = smem_u32(smem + C::kOffStages + slot * C::kStageBytes + C::kWBytes);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const uint64_t bdesc = smem_desc(xs + (uint32_t)((i & 1) * 2 + kk) * 32u, 16u, 1024u, 2u);
            const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
            if constexpr (C::kASmem) {
                // K-major, no swizzle: 8x16-byte core matrices, 128 B apart
                // along K, 512 B apart along rows; MMA kk starts 256 B in.
                const uint32_t as = smem_u32(smem + C::kOffA + aslot * C::kASlotBytes) + (uint32_t)kk * 256u;
                mma_smem_a(tmem_base + C::kDCol, smem_desc(as, 128u, 512u, 0u), bdesc, idesc, acc);
            } else {
                mma_tmem_a(tmem_base + C::kDCol, tmem_base + C::kACol + (uint32_t)(16 * aslot + 8 * kk), bdesc,
                           idesc, acc);
            }
        }
        mma_commit(b.aempty + aslot);
        if ((i & 1) == 1 || i == nchunks - 1) mma_commit(b.empty + slot);
    }
    if (failed) raise_timeout(p.status, abort_flag);
    mma_commit(b.accum);  // also fires when nothing was issued
    // before TMEM can be freed every issued MMA must have completed
    mma_commit(b.drain);
    mbar_wait(b.drain, 0, globaltimer_ns() + 1000000000ull);
}

// ------------------------------------------------------------------ decoders
template <class C>
__device__ void gemm_decode(const GemmParams &p, uint8_t *smem, const Bars &b, volatile uint32_t *abort_flag,
                            uint32_t tmem_base, int s0, int c0, int c1, uint64_t deadline) {
    const int q = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int r = threadIdx.x;  // row in the tile
    const int nchunks = c1 - c0;
    const uint8_t *hdr = smem + C::kOffHdr;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;

    if (!warp_wait(b.hdr, 0, deadline)) {
        if (lane == 0) raise_timeout(p.status, abort_flag);
        return;
    }
    Table T{};
    uint32_t mask_q = 0;
    const uint8_t *run = nullptr;
    int eslot = 0;
    for (int i = 0; i < nchunks; ++i) {
        if (warp_aborted(abort_flag)) return;
        const int chunk = c0 + i;
        const int jj = chunk & (kChunksPerSeg - 1);
        if (jj == 0) {
            const int ls = chunk / kChunksPerSeg - s0;
            const uint8_t *h = hdr + ls * kSegHdrBytes;
            T = make_table(*reinterpret_cast<const uint4 *>(h));
            const uint4 meta = *reinterpret_cast<const uint4 *>(h + 16);
            const uint32_t qc0 = meta.y & 0xFFFFu, qc1 = meta.y >> 16, qc2 = meta.z & 0xFFFFu, qc3 = meta.z >> 16;
            const uint32_t total = qc0 + qc1 + qc2 + qc3;
            const uint32_t qoff = (q > 0 ? qc0 : 0u) + (q > 1 ? qc1 : 0u) + (q > 2 ? qc2 : 0u);
            mask_q = (meta.w >> (8 * q)) & 0xFFu;
            eslot = ls & 1;
            if (!warp_wait(b.escfull + eslot, (uint32_t)(ls >> 1) & 1u, deadline)) {
                if (lane == 0) raise_timeout(p.status, abort_flag);
                return;
            }
            if (total > 0 && total + 30u <= (uint32_t)C::kEscCap)
                run = smem + C::kOffEsc + eslot * C::kEscCap + (meta.x & 15u) + qoff;
            else
                run = p.blob + p.off_esc + meta.x + qoff;
        }
        const int st = i >> 1, slot = st % C::kStages;
        if ((i & 1) == 0 && !warp_wait(b.full + slot, (uint32_t)(st / C::kStages) & 1u, deadline)) {
            if (lane == 0) raise_timeout(p.status, abort_flag);
            return;
        }
        const uint8_t *cp = smem + C::kOffStages + slot * C::kStageBytes + (i & 1) * kChunkBytes;
        const uint4 s_lo = *reinterpret_cast<const uint4 *>(cp + 16 * r);
        const uint4 s_hi = *reinterpret_cast<const uint4 *>(cp + kSlabBytes + 16 * r);
        const uint4 codes = *reinterpret_cast<const uint4 *>(cp + 2 * kSlabBytes + 16 * r);
        if ((i & 1) == 1 || i == nchunks - 1) {
            __syncwarp();
            if (lane == 0) mbar_arrive(b.empty + slot);  // this warp is done with the stage's bytes
        }
        uint32_t E[8];
        decode_exponents(T, codes, E);
        if ((mask_q >> jj) & 1u) run += warp_escapes(codes, run, E);
        uint32_t out[16];
        assemble(s_lo, s_hi, E, out);

        const int aslot = i % C::kASlots;
        if (i >= C::kASlots &&
            !warp_wait(b.aempty + aslot, (uint32_t)(i / C::kASlots - 1) & 1u, deadline)) {
            if (lane == 0) raise_timeout(p.status, abort_flag);
            return;
        }
        if constexpr (C::kASmem) {
            uint8_t *ap = smem + C::kOffA + aslot * C::kASlotBytes + (r >> 3) * 512 + (r & 7) * 16;
#pragma unroll
            for (int g = 0; g < 4; ++g)
                *reinterpret_cast<uint4 *>(ap + g * 128) =
                    make_uint4(out[4 * g], out[4 * g + 1], out[4 * g + 2], out[4 * g + 3]);
            fence_proxy_async_smem();
        } else {
            tc_fence_after();
            tmem_st16(tmem_base + lane_base + (uint32_t)(C::kACol + 16 * aslot), out);
            tmem_wait_st();
            tc_fence_before();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(b.afull + aslot);
        if (jj == kChunksPerSeg - 1 || i == nchunks - 1) {
            if (lane == 0) mbar_arrive(b.escempty + eslot);
        }
    }
}

// ------------------------------------------------------------------ epilogue
// D (fp32, TMEM lane = weight row, column = token) -> y, or -> partials and
// the last CTA of the tile sums the partials in split order.
template <class C>
__device__ void gemm_epilogue(const GemmParams &p, const Bars &b, volatile uint32_t *abort_flag,
                              volatile uint32_t *last_flag, uint32_t tmem_base, int64_t tile, int split,
                              uint64_t deadline) {
    const int q = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (warp_aborted(abort_flag)) return;
    if (!warp_wait(b.accum, 0, deadline)) {
        if (lane == 0) raise_timeout(p.status, abort_flag);
        return;
    }
    tc_fence_after();
    float acc[C::kNtok];
    {
        uint32_t v[16];
        tmem_ld16(tmem_base + ((uint32_t)(32 * q) << 16) + C::kDCol, v);
        tmem_wait_ld();
#pragma unroll
        for (int m = 0; m < 16; ++m) acc[m] = __uint_as_float(v[m]);
        if constexpr (C::kNtok == 32) {
            tmem_ld16(tmem_base + ((uint32_t)(32 * q) << 16) + C::kDCol + 16u, v);
            tmem_wait_ld();
#pragma unroll
            for (int m = 0; m < 16; ++m) acc[16 + m] = __uint_as_float(v[m]);
        }
    }
    const int64_t n = tile * kTileRows + 32 * q + lane;
    if (p.splits == 1) {
        if (n < p.N) {
#pragma unroll
            for (int m = 0; m < C::kNtok; ++m)
                if (m < p.M) p.y[(int64_t)m * p.N + n] = bf16_bits_rn(acc[m]);
        }
        return;
    }
    float *part = p.partials + (int64_t)split * p.M * p.Npad + n;
#pragma unroll
    for (int m = 0; m < C::kNtok; ++m)
        if (m < p.M) __stcg(part + (int64_t)m * p.Npad, acc[m]);
    __threadfence();
    // the four decode warps meet on mbarriers (bounded waits, no bar.sync that
    // a warp which gave up could leave the others stuck in)
    __syncwarp();
    if (lane == 0) mbar_arrive(b.epi_in);
    if (threadIdx.x == 0) {
        if (mbar_wait(b.epi_in, 0, deadline)) {
            __threadfence();
            const uint32_t old = atomicAdd(p.counters + tile, 1u);
            *last_flag = (old == (uint32_t)(p.splits - 1)) ? 1u : 0u;
            mbar_arrive(b.epi_out);
        } else {
            raise_timeout(p.status, abort_flag);
        }
    }
    if (!warp_wait(b.epi_out, 0, deadline)) {
        if (lane == 0) raise_timeout(p.status, abort_flag);
        return;
    }
    if (*last_flag == 0) return;
    __threadfence();
    if (n < p.N) {
#pragma unroll
        for (int m = 0; m < C::kNtok; ++m) {
            if (m < p.M) {
                float s = 0.0f;
                for (int sp = 0; sp < p.splits; ++sp)
                    s += __ldcg(p.partials + ((int64_t)sp * p.M + m) * p.Npad + n);
                p.y[(int64_t)m * p.N + n] = bf16_bits_rn(s);
            }
        }
    }
    if (threadIdx.x == 0) p.counters[tile] = 0u;  // ready for the next call
}

// ------------------------------------------------------------------ kernel
template <int NTOK, int STAGES, bool A_SMEM>
__global__ void __launch_bounds__(192, 1)
    w12_gemm_tc_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tmap_x) {
    using C = GemmCfg<NTOK, STAGES, A_SMEM>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBars);
    Bars b;
    b.full = bars;
    b.empty = b.full + STAGES;
    b.afull = b.empty + STAGES;
    b.aempty = b.afull + C::kASlots;
    b.escfull = b.aempty + C::kASlots;
    b.escempty = b.escfull + C::kEscSlots;
    b.hdr = b.escempty + C::kEscSlots;
    b.accum = b.hdr + 1;
    b.drain = b.accum + 1;
    b.epi_in = b.drain + 1;
    b.epi_out = b.epi_in + 1;
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    uint32_t *tmem_slot = misc;
    volatile uint32_t *abort_flag = misc + 1;
    volatile uint32_t *last_flag = misc + 2;

    const int warp = threadIdx.x >> 5;
    const int split = blockIdx.x;
    const int64_t tile = blockIdx.y;
    const int s0 = (int)((int64_t)split * p.segs / p.splits);
    const int s1 = (int)((int64_t)(split + 1) * p.segs / p.splits);
    const int c0 = s0 * kChunksPerSeg;
    const int c1 = min(s1 * kChunksPerSeg, p.chunks);
    const uint64_t deadline = globaltimer_ns() + p.timeout_ns;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(b.full + i, 1);
            mbar_init(b.empty + i, 4 + 1);
        }
        for (int i = 0; i < C::kASlots; ++i) {
            mbar_init(b.afull + i, 4);
            mbar_init(b.aempty + i, 1);
        }
        for (int i = 0; i < C::kEscSlots; ++i) {
            mbar_init(b.escfull + i, 1);
            mbar_init(b.escempty + i, 4);
        }
        mbar_init(b.hdr, 1);
        mbar_init(b.accum, 1);
        mbar_init(b.drain, 1);
        mbar_init(b.epi_in, 4);
        mbar_init(b.epi_out, 1);
        *abort_flag = 0u;
        *last_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 4) {
        if ((threadIdx.x & 31) == 0) gemm_producer<C>(p, &tmap_x, smem, b, abort_flag, tile, s0, c0, c1, deadline);
    } else if (warp == 5) {
        if ((threadIdx.x & 31) == 0) gemm_mma<C>(p, smem, b, abort_flag, tmem_base, c1 - c0, deadline);
        __syncwarp();
    } else {
        gemm_decode<C>(p, smem, b, abort_flag, tmem_base, s0, c0, c1, deadline);
        gemm_epilogue<C>(p, b, abort_flag, last_flag, tmem_base, tile, split, deadline);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem_base, C::kTmemCols);
}

}  // namespace dev
}  // namespace w12
