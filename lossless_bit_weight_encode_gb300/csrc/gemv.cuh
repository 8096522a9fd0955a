// W12 GEMV on CUDA cores (one or two tokens, M <= MT): y = x . W^T with W streamed from
// HBM in W12 form and decoded in registers ("decoded inside the GEMM
// registers", "SpecPilot: an agent doubled speculative decoding speed, and
// the 10.87x needs context", §The mechanisms it found; bit-exact weights,
// "StargazerX0/SpecPilot", §What it is).
//
// With one or two tokens the product is 2 or 4 flops per weight, far below
// what needs the tensor cores; what bounds this path is streaming the packed
// bytes and the integer decode.  So the decoded BF16 weights go straight into mixed
// precision fused multiply-adds (fma.rn.f32.bf16: BF16 weight times BF16 x
// into an fp32 sum, one per weight, on the FMA pipe) with no widening of
// either operand, no TMEM store and no handshake with an MMA warp.
//
// Warp roles (288 threads):
//   warps 0-7  decode: warp w handles rows 32q..32q+31 (q = w mod 4) and
//              columns 16h..16h+15 of every chunk (h = w / 4); per weight
//              stage (4 chunks) a thread reads its row's S bytes and codes from
//              SMEM, decodes 4 x 16 weights, patches escapes and accumulates
//              them against x (BF16 in SMEM, as the tensor TMA wrote it);
//   warp 8     producer: cp.async.bulk for the segment headers and every
//              weight stage (24 KB); per segment cp.async.bulk.tensor for the
//              256 x values and cp.async.bulk for the escape bytes.
// The two column halves of a row are added in fixed order at the end, then
// the split-K partials as in the tensor-core kernel.  Every wait is bounded.
#pragma once

#include "gemm_tc.cuh"

namespace w12 {
namespace dev {

template <int STAGES, int SCHUNKS, int MT>
struct GemvCfg {
    static constexpr int kMT = MT;                              // token rows of x (1 or 2)
    static constexpr int kThreads = 288;
    static constexpr int kDecWarps = 8;
    static constexpr int kStages = STAGES;
    static constexpr int kStageChunks = SCHUNKS;                // chunks per weight stage
    static constexpr int kStagesPerSeg = kChunksPerSeg / SCHUNKS;
    static constexpr int kWBytes = SCHUNKS * kChunkBytes;
    static constexpr int kXbBytes = MT * kSegK * 2;   // one segment of x, [MT][256] BF16 (TMA destination)
    static constexpr int kSegSlots = 2;
    static constexpr int kEscCap = 2048;
    static constexpr int kMaxSegs = 96;
    static constexpr int kOffW = 0;
    static constexpr int kOffXb = kOffW + STAGES * kWBytes;  // 128-byte aligned
    static constexpr int kOffEsc = kOffXb + kSegSlots * kXbBytes;
    static constexpr int kOffHdr = kOffEsc + kSegSlots * kEscCap;
    static constexpr int kOffRed = kOffHdr + kMaxSegs * kSegHdrBytes;  // [MT][128] fp32
    static constexpr int kOffBars = kOffRed + MT * kTileRows * 4;
    // wfull[S], wempty[S], sfull[2], sempty[2], hdr, red, epi_in, epi_out
    static constexpr int kNumBars = 2 * STAGES + 2 * kSegSlots + 4;
    static constexpr int kOffMisc = kOffBars + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 64 + 128;  // + slack to align the base to 128
    static_assert(kOffXb % 128 == 0, "TMA destination alignment");
    static_assert(kChunksPerSeg % SCHUNKS == 0, "stages must tile a segment");
};

struct GemvBars {
    uint64_t *wfull, *wempty, *sfull, *sempty, *hdr, *red, *epi_in, *epi_out;
};

// acc[t][j] += w * x[t] over 16 columns for each token t, with x as BF16 (16
// values per token at shared address xs + t * 512), one fma.rn.f32.bf16 per
// weight and token: the product of two BF16 values is exact in fp32, so this
// is the same single rounding as fma.rn.f32 on the widened operands.
// acc[t][j] collects the columns congruent to j mod 4.
template <int MT>
__device__ __forceinline__ void dot16_bf(const uint32_t (&w)[8], uint32_t xs, float (&acc)[MT][4]) {
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        const uint4 x0 = lds128(xs + (uint32_t)(t * kSegK * 2)), x1 = lds128(xs + (uint32_t)(t * kSegK * 2) + 16u);
        const uint32_t X[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
                "mov.b32 {wl, wh}, %4;\n\t"
                "mov.b32 {xl, xh}, %5;\n\t"
                "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
                "fma.rn.f32.bf16 %1, wh, xh, %1;\n\t"
                "mov.b32 {wl, wh}, %6;\n\t"
                "mov.b32 {xl, xh}, %7;\n\t"
                "fma.rn.f32.bf16 %2, wl, xl, %2;\n\t"
                "fma.rn.f32.bf16 %3, wh, xh, %3;\n\t}"
                : "+f"(acc[t][0]), "+f"(acc[t][1]), "+f"(acc[t][2]), "+f"(acc[t][3])
                : "r"(w[2 * g]), "r"(X[2 * g]), "r"(w[2 * g + 1]), "r"(X[2 * g + 1]));
        }
    }
}


// ------------------------------------------------------------------ producer
template <class C>
__device__ void gemv_producer(const GemmParams &p, const CUtensorMap *tmap, uint8_t *smem, const GemvBars &b,
                              volatile uint32_t *abort_flag, int64_t tile, int s0, int c0, int c1,
                              uint64_t deadline) {
    const int nchunks = c1 - c0;
    const int nsegs_cta = (nchunks + kChunksPerSeg - 1) / kChunksPerSeg;
    const int nstages = (nchunks + C::kStageChunks - 1) / C::kStageChunks;
    uint8_t *hdr = smem + C::kOffHdr;
    prefetch_tmap(tmap);

    const uint32_t hbytes = (uint32_t)nsegs_cta * kSegHdrBytes;
    mbar_arrive_expect_tx(b.hdr, hbytes);
    bulk_g2s(hdr, p.blob + p.off_seg + (uint64_t)(tile * p.segs + s0) * kSegHdrBytes, hbytes, b.hdr);
    bool hdr_ready = false;
    int issued = 0, seg_issued = 0;
    bool failed = false;

    for (int st = 0; st < nstages; ++st) {
        const int chunk = c0 + C::kStageChunks * st;
        // the stage's packed chunks first: they need nothing from the header
        const int slot = st % C::kStages;
        if (st >= C::kStages &&
            !mbar_wait(b.wempty + slot, (uint32_t)(st / C::kStages - 1) & 1u, deadline)) {
            failed = true;
            break;
        }
        const int nch = min(C::kStageChunks, c1 - chunk);
        mbar_arrive_expect_tx(b.wfull + slot, (uint32_t)(nch * kChunkBytes));
        bulk_g2s(smem + C::kOffW + slot * C::kWBytes,
                 p.blob + p.off_w + (uint64_t)(tile * p.chunks + chunk) * kChunkBytes, (uint32_t)(nch * kChunkBytes),
                 b.wfull + slot);
        issued = st + 1;
        if ((chunk & (kChunksPerSeg - 1)) == 0) {
            // a segment starts: its x (no header needed), then its escapes;
            // the one arrival comes last so the phase cannot complete early
            const int ls = chunk / kChunksPerSeg - s0;
            const int sslot = ls & 1;
            if (ls >= 2 && !mbar_wait(b.sempty + sslot, (uint32_t)((ls >> 1) - 1) & 1u, deadline)) {
                failed = true;
                break;
            }
            mbar_expect_tx(b.sfull + sslot, (uint32_t)C::kXbBytes);
            tma_load_2d(smem + C::kOffXb + sslot * C::kXbBytes, tmap, chunk * kChunkK, 0, b.sfull + sslot);
            seg_issued = ls + 1;
            if (!hdr_ready) {
                if (!mbar_wait(b.hdr, 0, deadline)) { failed = true; break; }
                hdr_ready = true;
            }
            const uint4 meta = *reinterpret_cast<const uint4 *>(hdr + ls * kSegHdrBytes + 16);
            const uint32_t base = meta.x;
            const uint32_t total = seg_escape_total(meta);
            if (escapes_staged<C>(total)) {
                const uint32_t src0 = base & ~15u;
                const uint32_t ebytes = ((base + total + 15u) & ~15u) - src0;
                mbar_expect_tx(b.sfull + sslot, ebytes);
                bulk_g2s(smem + C::kOffEsc + sslot * C::kEscCap, p.blob + p.off_esc + src0, ebytes, b.sfull + sslot);
            }
            mbar_arrive(b.sfull + sslot);
        }
        if (*abort_flag) break;
    }
    if (failed) raise_timeout(p.status, abort_flag);
    if (*abort_flag) {
        const uint64_t drain_deadline = globaltimer_ns() + 1000000000ull;
        for (int st = max(0, issued - C::kStages); st < issued; ++st)
            mbar_wait(b.wfull + st % C::kStages, (uint32_t)(st / C::kStages) & 1u, drain_deadline);
        for (int ls = max(0, seg_issued - 2); ls < seg_issued; ++ls)
            mbar_wait(b.sfull + (ls & 1), (uint32_t)(ls >> 1) & 1u, drain_deadline);
        mbar_wait(b.hdr, 0, drain_deadline);
    }
}

// ------------------------------------------------------------------ decoders
template <class C>
__device__ void gemv_decode(const GemmParams &p, uint8_t *smem, const GemvBars &b, volatile uint32_t *abort_flag,
                            volatile uint32_t *last_flag, int64_t tile, int split, int s0, int c0, int c1,
                            uint64_t deadline) {
    const int warp = threadIdx.x >> 5;
    const int q = warp & 3;       // rows 32q..32q+31
    const int h = warp >> 2;      // columns 16h..16h+15 of each chunk
    const int lane = threadIdx.x & 31;
    const int r = 32 * q + lane;  // row in the tile
    const int nchunks = c1 - c0;
    const int nstages = (nchunks + C::kStageChunks - 1) / C::kStageChunks;
    const uint8_t *hdr = smem + C::kOffHdr;
    const uint32_t s_row = smem_u32(smem + C::kOffW) + (uint32_t)(h * kSlabBytes + 16 * r);
    const uint32_t c_off = (uint32_t)((2 - h) * kSlabBytes);
    const uint32_t xb0 = smem_u32(smem + C::kOffXb) + (uint32_t)(16 * h) * 2u;

    float acc[C::kMT][4];
#pragma unroll
    for (int t = 0; t < C::kMT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
    bool ok = warp_wait(b.hdr, 0, deadline);
    Table T{};
    uint32_t mask_q = 0, xseg = 0;
    const uint8_t *run = nullptr;
    for (int st = 0; ok && st < nstages; ++st) {
        const int chunk0 = c0 + C::kStageChunks * st;
        const int jj0 = chunk0 & (kChunksPerSeg - 1);
        const int ls = st / C::kStagesPerSeg;
        const int sslot = ls & 1;
        const int nch = min(C::kStageChunks, c1 - chunk0);
        if (jj0 == 0) {
            const uint8_t *hp = hdr + (chunk0 / kChunksPerSeg - s0) * kSegHdrBytes;
            T = make_table(*reinterpret_cast<const uint4 *>(hp));
            const uint4 meta = *reinterpret_cast<const uint4 *>(hp + 16);
            const uint32_t qc0 = meta.y & 0xFFFFu, qc1 = meta.y >> 16, qc2 = meta.z & 0xFFFFu;
            const uint32_t qoff = (q > 0 ? qc0 : 0u) + (q > 1 ? qc1 : 0u) + (q > 2 ? qc2 : 0u);
            mask_q = (meta.w >> (8 * q)) & 0xFFu;
            if (!(ok = warp_wait(b.sfull + sslot, (uint32_t)(ls >> 1) & 1u, deadline))) break;
            if (escapes_staged<C>(seg_escape_total(meta)))
                run = smem + C::kOffEsc + sslot * C::kEscCap + (meta.x & 15u) + qoff;
            else
                run = p.blob + p.off_esc + meta.x + qoff;
            xseg = xb0 + (uint32_t)(sslot * C::kXbBytes);
        }
        const int slot = st % C::kStages;
        if (!(ok = warp_wait(b.wfull + slot, (uint32_t)(st / C::kStages) & 1u, deadline))) break;
        // read the whole stage first so that its slot is freed early
        const uint32_t sa = s_row + (uint32_t)(slot * C::kWBytes);
        uint4 sb[C::kStageChunks], cd[C::kStageChunks];
#pragma unroll
        for (int e = 0; e < C::kStageChunks; ++e) {
            if (e < nch) {
                sb[e] = lds128(sa + (uint32_t)(e * kChunkBytes));
                cd[e] = lds128(sa + (uint32_t)(e * kChunkBytes) + c_off);
            }
        }
        warp_arrive(b.wempty + slot);

        const uint32_t stage_esc = (mask_q >> jj0) & ((1u << C::kStageChunks) - 1u);
        if (nch == C::kStageChunks && stage_esc == 0) {
            // common case, decided once per stage for the whole warp: a full
            // stage without escapes
#pragma unroll
            for (int e = 0; e < C::kStageChunks; ++e) {
                uint32_t E[4], out[8];
                decode_exponents_half(T, h ? cd[e].z : cd[e].x, h ? cd[e].w : cd[e].y, E);
                assemble_half(sb[e], E, out);
                dot16_bf<C::kMT>(out, xseg + (uint32_t)((jj0 + e) * kChunkK * 2), acc);
            }
        } else {
#pragma unroll
            for (int e = 0; e < C::kStageChunks; ++e) {
                if (e < nch) {
                    uint32_t out[8];
                    decode_half_chunk(T, sb[e], cd[e], h, (stage_esc >> e) & 1u, run, out);
                    dot16_bf<C::kMT>(out, xseg + (uint32_t)((jj0 + e) * kChunkK * 2), acc);
                }
            }
        }
        if (jj0 + nch == kChunksPerSeg || st == nstages - 1) {
            warp_arrive(b.sempty + sslot);  // done with this segment's x and escapes
        }
    }
    if (!ok) {
        if (lane == 0) raise_timeout(p.status, abort_flag);
        return;
    }

    // ---- epilogue: add the two column halves of each row in fixed order
    constexpr int MT = C::kMT;
    float mine[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) mine[t] = (acc[t][0] + acc[t][1]) + (acc[t][2] + acc[t][3]);
    float *red = reinterpret_cast<float *>(smem + C::kOffRed);
    if (h == 1) {
#pragma unroll
        for (int t = 0; t < MT; ++t) red[t * kTileRows + r] = mine[t];
        __syncwarp();
        if (lane == 0) mbar_arrive(b.red);
        return;
    }
    if (!warp_wait(b.red, 0, deadline)) {
        if (lane == 0) raise_timeout(p.status, abort_flag);
        return;
    }
    float total[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) total[t] = mine[t] + red[t * kTileRows + r];
    const int64_t n = tile * kTileRows + r;
    if (p.splits == 1) {
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            if (t < p.M) {
                if (p.y != nullptr && n < p.N) p.y[(int64_t)t * p.N + n] = bf16_bits_rn(total[t]);
                if (p.amax != nullptr) argmax_warp(p.amax + t, n < p.N ? argmax_key(total[t], (uint32_t)n) : 0ull);
            }
        }
        return;
    }
#pragma unroll
    for (int t = 0; t < MT; ++t)
        if (t < p.M) __stcg(p.partials + ((int64_t)split * p.M + t) * p.Npad + n, total[t]);
    // the mbarrier arrive/wait pair orders these stores before thread 0's
    // release increment of the tile counter, which publishes them all
    __syncwarp();
    if (lane == 0) mbar_arrive(b.epi_in);
    if (threadIdx.x == 0) {
        if (mbar_wait(b.epi_in, 0, deadline)) {
            const uint32_t old = arrive_acq_rel(p.counters + tile);
            const bool last = old == (uint32_t)(p.splits - 1);
            *last_flag = last ? 1u : 0u;
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
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        if (t >= p.M) continue;
        // ascending split order; eight loads in flight at a time
        const float *src = p.partials + (int64_t)t * p.Npad + (n < p.N ? n : tile * kTileRows);
        const int64_t stride = (int64_t)p.M * p.Npad;
        float s = 0.0f;
        int sp = 0;
        for (; sp + 8 <= p.splits; sp += 8) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldcg(src + (int64_t)(sp + u) * stride);
#pragma unroll
            for (int u = 0; u < 8; ++u) s += v[u];
        }
        for (; sp < p.splits; ++sp) s += __ldcg(src + (int64_t)sp * stride);
        if (p.y != nullptr && n < p.N) p.y[(int64_t)t * p.N + n] = bf16_bits_rn(s);
        if (p.amax != nullptr) argmax_warp(p.amax + t, n < p.N ? argmax_key(s, (uint32_t)n) : 0ull);
    }
    if (threadIdx.x == 0) p.counters[tile] = 0u;  // ready for the next call
}

// ------------------------------------------------------------------ kernel
template <int STAGES, int SCHUNKS, int MT>
__global__ void __launch_bounds__(288, 2)
    w12_gemv_kernel(const __grid_constant__ GemmGroup grp, const __grid_constant__ CUtensorMap tmap_x) {
    using C = GemvCfg<STAGES, SCHUNKS, MT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBars);
    GemvBars b;
    b.wfull = bars;
    b.wempty = b.wfull + STAGES;
    b.sfull = b.wempty + STAGES;
    b.sempty = b.sfull + C::kSegSlots;
    b.hdr = b.sempty + C::kSegSlots;
    b.red = b.hdr + 1;
    b.epi_in = b.red + 1;
    b.epi_out = b.epi_in + 1;
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile uint32_t *abort_flag = misc + 1;
    volatile uint32_t *last_flag = misc + 2;

    const int warp = threadIdx.x >> 5;
    const int split = blockIdx.x;
    int64_t tile;
    const GemmParams &p = grp.m[group_member(grp, &tile)];
    const int s0 = (int)((int64_t)split * p.segs / p.splits);
    const int s1 = (int)((int64_t)(split + 1) * p.segs / p.splits);
    const int c0 = s0 * kChunksPerSeg;
    const int c1 = min(s1 * kChunksPerSeg, p.chunks);
    const uint64_t deadline = globaltimer_ns() + p.timeout_ns;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(b.wfull + i, 1);
            mbar_init(b.wempty + i, C::kDecWarps);
        }
        for (int i = 0; i < C::kSegSlots; ++i) {
            mbar_init(b.sfull + i, 1);
            mbar_init(b.sempty + i, C::kDecWarps);
        }
        mbar_init(b.hdr, 1);
        mbar_init(b.red, 4);
        mbar_init(b.epi_in, 4);
        mbar_init(b.epi_out, 1);
        *abort_flag = 0u;
        *last_flag = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) pdl_launch_dependents();
    if (warp == 8 && (threadIdx.x & 31) == 0) prefetch_cta_weights<kChunkBytes, true>(p, tile, s0, c0, c1);
    pdl_wait();
    if (warp == 8) {
        if ((threadIdx.x & 31) == 0) gemv_producer<C>(p, &tmap_x, smem, b, abort_flag, tile, s0, c0, c1, deadline);
    } else {
        gemv_decode<C>(p, smem, b, abort_flag, last_flag, tile, split, s0, c0, c1, deadline);
    }
}

}  // namespace dev
}  // namespace w12
