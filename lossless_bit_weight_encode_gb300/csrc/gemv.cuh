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
    // wfull[S], wempty[S], sfull[2], sempty[2], hdr, red, red_empty, epi_in, epi_out
    static constexpr int kNumBars = 2 * STAGES + 2 * kSegSlots + 5;
    static constexpr int kOffMisc = kOffBars + kNumBars * 8;
    static constexpr int kMaxPieces = 2;                        // pieces of one CTA's work
    static constexpr int kOffPieces = kOffMisc + 64;
    static constexpr int kSmemBytes = kOffPieces + kMaxPieces * (int)sizeof(Piece) + 128;  // + base alignment slack
    static_assert(kOffXb % 128 == 0, "TMA destination alignment");
    static_assert(kChunksPerSeg % SCHUNKS == 0, "stages must tile a segment");
};

struct GemvBars {
    uint64_t *wfull, *wempty, *sfull, *sempty, *hdr, *red, *red_empty, *epi_in, *epi_out;
    uint64_t *first_done, *prod_done;  // used by the one-CTA-per-SM kernel only
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
// Stage and segment counters run on across the CTA's pieces, so the ring
// slots and mbarrier phases continue from one tile to the next.
template <class C>
__device__ void gemv_producer(const GemmGroup &g, const Piece *pieces, int npieces, const CUtensorMap *tmap,
                              uint8_t *smem, const GemvBars &b, volatile uint32_t *abort_flag, uint64_t deadline) {
    uint8_t *hdr = smem + C::kOffHdr;
    prefetch_tmap(tmap);

    // the segment headers of every piece, one after another, on one phase
    uint32_t hbytes = 0;
    for (int k = 0; k < npieces; ++k) hbytes += (uint32_t)(pieces[k].s1 - pieces[k].s0) * kSegHdrBytes;
    mbar_arrive_expect_tx(b.hdr, hbytes);
    for (int k = 0, off = 0; k < npieces; ++k) {
        const Piece &pc = pieces[k];
        const GemmParams &p = g.m[pc.member];
        const uint32_t n = (uint32_t)(pc.s1 - pc.s0) * kSegHdrBytes;
        bulk_g2s(hdr + off, p.blob + p.off_seg + (uint64_t)(pc.tile * p.segs + pc.s0) * kSegHdrBytes, n, b.hdr);
        off += (int)n;
    }

    bool hdr_ready = false, failed = false, stop = false;
    int gst = 0, gls = 0;  // weight stages and segments issued
    int hseg = 0;          // headers of the earlier pieces
    for (int k = 0; !stop && k < npieces; ++k) {
        const Piece &pc = pieces[k];
        const GemmParams &p = g.m[pc.member];
        const int c0 = pc.s0 * kChunksPerSeg, c1 = min(pc.s1 * kChunksPerSeg, p.chunks);
        const int nstages = (c1 - c0 + C::kStageChunks - 1) / C::kStageChunks;
        for (int st = 0; st < nstages; ++st) {
            const int chunk = c0 + C::kStageChunks * st;
            // the stage's packed chunks first: they need nothing from the header
            const int slot = gst % C::kStages;
            if (gst >= C::kStages &&
                !mbar_wait(b.wempty + slot, (uint32_t)(gst / C::kStages - 1) & 1u, deadline)) {
                failed = stop = true;
                break;
            }
            const int nch = min(C::kStageChunks, c1 - chunk);
            mbar_arrive_expect_tx(b.wfull + slot, (uint32_t)(nch * kChunkBytes));
            bulk_g2s(smem + C::kOffW + slot * C::kWBytes,
                     p.blob + p.off_w + (uint64_t)(pc.tile * p.chunks + chunk) * kChunkBytes,
                     (uint32_t)(nch * kChunkBytes), b.wfull + slot);
            ++gst;
            if ((chunk & (kChunksPerSeg - 1)) == 0) {
                // a segment starts: its x (no header needed), then its escapes;
                // the one arrival comes last so the phase cannot complete early
                const int ls = chunk / kChunksPerSeg - pc.s0;
                const int sslot = gls & 1;
                if (gls >= 2 && !mbar_wait(b.sempty + sslot, (uint32_t)((gls >> 1) - 1) & 1u, deadline)) {
                    failed = stop = true;
                    break;
                }
                mbar_expect_tx(b.sfull + sslot, (uint32_t)C::kXbBytes);
                tma_load_2d(smem + C::kOffXb + sslot * C::kXbBytes, tmap, chunk * kChunkK, 0, b.sfull + sslot);
                ++gls;
                if (!hdr_ready) {
                    if (!mbar_wait(b.hdr, 0, deadline)) {
                        mbar_arrive(b.sfull + sslot);  // lets the phase end once x has landed
                        failed = stop = true;
                        break;
                    }
                    hdr_ready = true;
                }
                const uint4 meta = *reinterpret_cast<const uint4 *>(hdr + (hseg + ls) * kSegHdrBytes + 16);
                const uint32_t base = meta.x;
                const uint32_t total = seg_escape_total(meta);
                if (escapes_staged<C>(total)) {
                    const uint32_t src0 = base & ~15u;
                    const uint32_t ebytes = ((base + total + 15u) & ~15u) - src0;
                    mbar_expect_tx(b.sfull + sslot, ebytes);
                    bulk_g2s(smem + C::kOffEsc + sslot * C::kEscCap, p.blob + p.off_esc + src0, ebytes,
                             b.sfull + sslot);
                }
                mbar_arrive(b.sfull + sslot);
            }
            if (*abort_flag) {
                stop = true;
                break;
            }
        }
        hseg += pc.s1 - pc.s0;
    }
    if (failed) raise_timeout(group_status(g), abort_flag);
    if (*abort_flag) {
        const uint64_t drain_deadline = globaltimer_ns() + 1000000000ull;
        for (int st = max(0, gst - C::kStages); st < gst; ++st)
            mbar_wait(b.wfull + st % C::kStages, (uint32_t)(st / C::kStages) & 1u, drain_deadline);
        for (int ls = max(0, gls - 2); ls < gls; ++ls)
            mbar_wait(b.sfull + (ls & 1), (uint32_t)(ls >> 1) & 1u, drain_deadline);
        mbar_wait(b.hdr, 0, drain_deadline);
    }
}

// ------------------------------------------------------------------ decoders
// Per piece: decode and accumulate its stages, then add the two column halves
// of each row (h = 1 hands its sums to h = 0 through shared memory) and write
// the whole tile's result when the CTA owns the tile, else the piece's
// partial-sum slot.  After the last piece: one arrival on the counter of each
// shared tile; the last arrival adds the tile's slots in slot order.
template <class C>
__device__ void gemv_decode(const GemmGroup &g, const Piece *pieces, int npieces, uint8_t *smem, const GemvBars &b,
                            volatile uint32_t *abort_flag, volatile uint32_t *last_flags, uint64_t deadline) {
    constexpr int MT = C::kMT;
    const int warp = threadIdx.x >> 5;
    const int q = warp & 3;       // rows 32q..32q+31
    const int h = warp >> 2;      // columns 16h..16h+15 of each chunk
    const int lane = threadIdx.x & 31;
    const int r = 32 * q + lane;  // row in the tile
    const uint8_t *hdr = smem + C::kOffHdr;
    const uint32_t s_row = smem_u32(smem + C::kOffW) + (uint32_t)(h * kSlabBytes + 16 * r);
    const uint32_t c_off = (uint32_t)((2 - h) * kSlabBytes);
    const uint32_t xb0 = smem_u32(smem + C::kOffXb) + (uint32_t)(16 * h) * 2u;
    float *red = reinterpret_cast<float *>(smem + C::kOffRed);

    bool ok = warp_wait(b.hdr, 0, deadline);
    int gst = 0, gls = 0;  // weight stages and segments consumed
    int hseg = 0;          // headers of the earlier pieces
    uint32_t shared = 0;   // pieces whose partial sums went to a split-K slot
    for (int k = 0; ok && k < npieces; ++k) {
        const Piece &pc = pieces[k];
        const GemmParams &p = g.m[pc.member];
        const int c0 = pc.s0 * kChunksPerSeg, c1 = min(pc.s1 * kChunksPerSeg, p.chunks);
        const int nstages = (c1 - c0 + C::kStageChunks - 1) / C::kStageChunks;
        float acc[MT][4];
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
        Table T{};
        uint32_t mask_q = 0, xseg = 0;
        int sslot = 0;
        const uint8_t *run = nullptr;
        for (int st = 0; st < nstages; ++st) {
            const int chunk0 = c0 + C::kStageChunks * st;
            const int jj0 = chunk0 & (kChunksPerSeg - 1);
            const int nch = min(C::kStageChunks, c1 - chunk0);
            if (jj0 == 0) {
                const uint8_t *hp = hdr + (hseg + st / C::kStagesPerSeg) * kSegHdrBytes;
                T = make_table(*reinterpret_cast<const uint4 *>(hp));
                const uint4 meta = *reinterpret_cast<const uint4 *>(hp + 16);
                const uint32_t qc0 = meta.y & 0xFFFFu, qc1 = meta.y >> 16, qc2 = meta.z & 0xFFFFu;
                const uint32_t qoff = (q > 0 ? qc0 : 0u) + (q > 1 ? qc1 : 0u) + (q > 2 ? qc2 : 0u);
                mask_q = (meta.w >> (8 * q)) & 0xFFu;
                sslot = gls & 1;
                if (!(ok = warp_wait(b.sfull + sslot, (uint32_t)(gls >> 1) & 1u, deadline))) break;
                ++gls;
                if (escapes_staged<C>(seg_escape_total(meta)))
                    run = smem + C::kOffEsc + sslot * C::kEscCap + (meta.x & 15u) + qoff;
                else
                    run = p.blob + p.off_esc + meta.x + qoff;
                xseg = xb0 + (uint32_t)(sslot * C::kXbBytes);
            }
            const int slot = gst % C::kStages;
            if (!(ok = warp_wait(b.wfull + slot, (uint32_t)(gst / C::kStages) & 1u, deadline))) break;
            ++gst;
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
                    dot16_bf<MT>(out, xseg + (uint32_t)((jj0 + e) * kChunkK * 2), acc);
                }
            } else {
#pragma unroll
                for (int e = 0; e < C::kStageChunks; ++e) {
                    if (e < nch) {
                        uint32_t out[8];
                        decode_half_chunk(T, sb[e], cd[e], h, (stage_esc >> e) & 1u, run, out);
                        dot16_bf<MT>(out, xseg + (uint32_t)((jj0 + e) * kChunkK * 2), acc);
                    }
                }
            }
            if (jj0 + nch == kChunksPerSeg || st == nstages - 1) {
                warp_arrive(b.sempty + sslot);  // done with this segment's x and escapes
            }
        }
        if (!ok) break;
        hseg += pc.s1 - pc.s0;

        // ---- add the two column halves of each row in fixed order
        float mine[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) mine[t] = (acc[t][0] + acc[t][1]) + (acc[t][2] + acc[t][3]);
        if (h == 1) {
            // the buffer is free once h = 0 has read the previous piece's sums
            if (k > 0 && !(ok = warp_wait(b.red_empty, (uint32_t)(k - 1) & 1u, deadline))) break;
#pragma unroll
            for (int t = 0; t < MT; ++t) red[t * kTileRows + r] = mine[t];
            __syncwarp();
            if (lane == 0) mbar_arrive(b.red);
            continue;
        }
        if (!(ok = warp_wait(b.red, (uint32_t)k & 1u, deadline))) break;
        float total[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) total[t] = mine[t] + red[t * kTileRows + r];
        __syncwarp();
        if (lane == 0) mbar_arrive(b.red_empty);
        const int64_t n = pc.tile * kTileRows + r;
        if (pc.count == 1) {
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                if (t < p.M) {
                    if (p.y != nullptr && n < p.N) p.y[(int64_t)t * p.N + n] = bf16_bits_rn(total[t]);
                    if (p.amax != nullptr)
                        argmax_warp(p.amax + t, n < p.N ? argmax_key(total[t], (uint32_t)n) : 0ull);
                }
            }
            continue;
        }
#pragma unroll
        for (int t = 0; t < MT; ++t)
            if (t < p.M) __stcg(p.partials + ((int64_t)pc.idx * p.M + t) * p.Npad + n, total[t]);
        shared |= 1u << k;
    }
    if (!ok) {
        if (lane == 0) raise_timeout(group_status(g), abort_flag);
        return;
    }
    if (h == 1 || shared == 0) return;

    // ---- split-K arrivals of the pieces whose tile other CTAs share, once at
    // the end so that no piece boundary waits for an atomic; the mbarrier
    // arrive/wait pair orders every partial store before thread 0's release
    // fence, which with the increments after it publishes them
    __syncwarp();
    if (lane == 0) mbar_arrive(b.epi_in);
    if (threadIdx.x == 0) {
        if (mbar_wait(b.epi_in, 0, deadline)) {
            uint32_t old[C::kMaxPieces];
            fence_acq_rel_gpu();
#pragma unroll
            for (int k = 0; k < C::kMaxPieces; ++k)
                if (k < npieces && ((shared >> k) & 1u))
                    old[k] = arrive_relaxed(g.m[pieces[k].member].counters + pieces[k].tile);
            bool any_last = false;
#pragma unroll
            for (int k = 0; k < C::kMaxPieces; ++k) {
                if (k < npieces && ((shared >> k) & 1u)) {
                    const bool last = old[k] == (uint32_t)(pieces[k].count - 1);
                    last_flags[k] = last ? 1u : 0u;
                    any_last |= last;
                }
            }
            if (any_last) fence_acq_rel_gpu();
            mbar_arrive(b.epi_out);
        } else {
            raise_timeout(group_status(g), abort_flag);
        }
    }
    if (!warp_wait(b.epi_out, 0, deadline)) {
        if (lane == 0) raise_timeout(group_status(g), abort_flag);
        return;
    }
    for (int k = 0; k < npieces; ++k) {
        if (!((shared >> k) & 1u) || last_flags[k] == 0) continue;
        // the last arrival adds the tile's slots in ascending order, eight
        // loads in flight at a time
        const Piece &pc = pieces[k];
        const GemmParams &p = g.m[pc.member];
        const int64_t n = pc.tile * kTileRows + r;
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            if (t >= p.M) continue;
            const float *src = p.partials + (int64_t)t * p.Npad + (n < p.N ? n : pc.tile * kTileRows);
            const int64_t stride = (int64_t)p.M * p.Npad;
            float s = 0.0f;
            for (int sp = 0; sp < pc.count; sp += 8) {
                // up to eight slots loaded at once, added in slot order
                float v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (sp + u < pc.count) v[u] = __ldcg(src + (int64_t)(sp + u) * stride);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (sp + u < pc.count) s += v[u];
            }
            if (p.y != nullptr && n < p.N) p.y[(int64_t)t * p.N + n] = bf16_bits_rn(s);
            if (p.amax != nullptr) argmax_warp(p.amax + t, n < p.N ? argmax_key(s, (uint32_t)n) : 0ull);
        }
        if (threadIdx.x == 0) p.counters[pc.tile] = 0u;  // ready for the next call
    }
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
    b.red_empty = b.red + 1;
    b.epi_in = b.red_empty + 1;
    b.epi_out = b.epi_in + 1;
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile uint32_t *abort_flag = misc + 1;
    volatile uint32_t *npieces = misc + 2;
    volatile uint32_t *last_flags = misc + 4;  // [kMaxPieces]
    Piece *pieces = reinterpret_cast<Piece *>(smem + C::kOffPieces);

    const int warp = threadIdx.x >> 5;
    const uint64_t deadline = globaltimer_ns() + grp.m[0].timeout_ns;

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
        mbar_init(b.red_empty, 4);
        mbar_init(b.epi_in, 4);
        mbar_init(b.epi_out, 1);
        *abort_flag = 0u;
        // this CTA's pieces: one with fixed split-K; with stream-K a range of
        // at most segs units (a single wave of more CTAs than tiles), so at
        // most two tiles
        CtaWork w = cta_work(grp);
        uint32_t n = 0;
        while (n < C::kMaxPieces && next_piece(grp, w, pieces[n])) ++n;
        *npieces = n;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) pdl_launch_dependents();
    const int np = (int)*npieces;
    if (warp == 8 && (threadIdx.x & 31) == 0) prefetch_pieces<kChunkBytes, true>(grp, pieces, np);
    pdl_wait();
    if (warp == 8) {
        if ((threadIdx.x & 31) == 0) gemv_producer<C>(grp, pieces, np, &tmap_x, smem, b, abort_flag, deadline);
    } else {
        gemv_decode<C>(grp, pieces, np, smem, b, abort_flag, last_flags, deadline);
    }
}

}  // namespace dev
}  // namespace w12
