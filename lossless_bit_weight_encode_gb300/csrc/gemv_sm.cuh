// W12 GEMV on CUDA cores, one CTA per SM (one or two tokens, M <= MT): y =
// x . W^T with W streamed from HBM in W12 form and decoded in registers
// ("decoded inside the GEMM registers", "SpecPilot: an agent doubled
// speculative decoding speed, and the 10.87x needs context", §The mechanisms
// it found; bit-exact weights, "StargazerX0/SpecPilot", §What it is).
//
// The arithmetic is that of the two-CTA kernel in gemv.cuh (the same decode,
// the same fma.rn.f32.bf16 per weight and token); what differs is how an SM's
// warps share the work.  Two independent CTAs per SM do not finish together:
// the warps of the CTA placed first win issue priority, so it ends its share
// early and the other CTA runs its last stretch alone, with half the warps,
// at about 70 % of the SM's two-CTA rate.  Here all sixteen decode warps of an
// SM consume one weight stage (a whole 256-column segment) together, so none
// can run ahead of the others by more than the ring's depth and the SM keeps
// every warp busy to the end of its work.
//
// Warp roles (544 threads):
//   warps 0-15  decode: warp w handles rows 32q..32q+31 (q = w mod 4) and
//               chunks 2j, 2j+1 of each segment (j = w / 4), both column
//               halves; per stage a thread reads its row's S bytes and codes of
//               its two chunks from SMEM, decodes 64 weights, patches escapes
//               and accumulates them against x (BF16 in SMEM, as the tensor TMA
//               wrote it);
//   warp 16     producer: cp.async.bulk for the segment headers and every
//               weight stage (48 KB); per segment cp.async.bulk.tensor for the
//               256 x values and cp.async.bulk for the escape bytes.
// The four chunk groups of a row are added in fixed order at the end of each
// piece, then split-K as in gemv.cuh.  Every wait is bounded.
#pragma once

#include "gemv.cuh"

namespace w12 {
namespace dev {

template <int MT>
struct GemvSmCfg {
    static constexpr int kMT = MT;                              // token rows of x (1 or 2)
    static constexpr int kDecWarps = 16;
    static constexpr int kThreads = (kDecWarps + 1) * 32;
    static constexpr int kStages = 4;
    static constexpr int kWBytes = kChunksPerSeg * kChunkBytes;  // one segment per stage
    static constexpr int kXbBytes = MT * kSegK * 2;             // one segment of x, [MT][256] BF16
    // x + escape slots, one segment each, as deep as the weight ring: with two
    // the producer waited for the consumers before issuing the weights four
    // stages ahead (measured 113.8 us per layer step at M = 1 against 109.9
    // with four; five or six were slower again)
    static constexpr int kSegSlots = 4;
    static constexpr int kEscCap = 2048;
    static constexpr int kMaxSegs = 256;                        // units (segments) of one CTA
    static constexpr int kMaxPieces = 64;                       // tiles one CTA's range meets
    static constexpr int kOffW = 0;
    static constexpr int kOffXb = kOffW + kStages * kWBytes;    // 128-byte aligned
    static constexpr int kOffEsc = kOffXb + kSegSlots * kXbBytes;
    static constexpr int kOffHdr = kOffEsc + kSegSlots * kEscCap;
    static constexpr int kOffRed = kOffHdr + kMaxSegs * kSegHdrBytes;  // [3][MT][128] fp32
    static constexpr int kOffBars = kOffRed + 3 * MT * kTileRows * 4;
    // wfull[S], wempty[S], sfull[S], sempty[S], hdr, red, red_empty, epi_in,
    // epi_out, first_done, prod_done
    static constexpr int kNumBars = 2 * kStages + 2 * kSegSlots + 7;
    static constexpr int kOffMisc = kOffBars + kNumBars * 8;
    static constexpr int kOffPieces = kOffMisc + 64;
    static constexpr int kSmemBytes = kOffPieces + kMaxPieces * (int)sizeof(Piece) + 128;  // + base alignment slack
    static_assert(kOffXb % 128 == 0, "TMA destination alignment");
    static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM must fit");
};

// Escapes in quarter-chunk (rows of this warp) whose codes this thread's row
// holds in cd: the warp total, the same on every lane.
__device__ __forceinline__ uint32_t chunk_escapes(const uint4 &cd) {
    const uint32_t n = __popc(escape_flags(cd.x)) + __popc(escape_flags(cd.y)) + __popc(escape_flags(cd.z)) +
                       __popc(escape_flags(cd.w));
    return __reduce_add_sync(0xFFFFFFFFu, n);
}

// Where the escapes of chunk 2j of quarter q start in the segment's escape
// run, relative to the run's first byte, for a warp that decodes chunks 2j
// and 2j + 1 of a segment staged at shared address sw + 16 * row (this
// thread's row).  The run orders a quarter's escapes chunk by chunk and the
// header holds only each quarter's total, so the warp counts escape codes:
// of the earlier chunks (j < 2), or of its own and the later chunks, taken
// from the quarter's total (j >= 2) -- whichever end has fewer chunks; the
// segment's mask skips chunks without escapes.  acd / bcd are the codes of
// the warp's chunks, esc_a / esc_b whether they hold escapes.
__device__ __forceinline__ uint32_t quarter_chunk_escape_pos(const uint4 &meta, int q, int j, uint32_t mask_q,
                                                             int nch, const uint4 &acd, const uint4 &bcd,
                                                             uint32_t esc_a, uint32_t esc_b, uint32_t sw) {
    const uint32_t qc0 = meta.y & 0xFFFFu, qc1 = meta.y >> 16, qc2 = meta.z & 0xFFFFu;
    const uint32_t qc_mine = ((q < 2 ? meta.y : meta.z) >> (16 * (q & 1))) & 0xFFFFu;
    uint32_t pos = (q > 0 ? qc0 : 0u) + (q > 1 ? qc1 : 0u) + (q > 2 ? qc2 : 0u);
    const int ca = 2 * j;
    if (j < 2) {
        for (int c = 0; c < ca; ++c)
            if ((mask_q >> c) & 1u) pos += chunk_escapes(lds128(sw + (uint32_t)(c * kChunkBytes) + 2u * kSlabBytes));
        return pos;
    }
    uint32_t after = 0;
    if (esc_a) after += chunk_escapes(acd);
    if (esc_b) after += chunk_escapes(bcd);
    for (int c = ca + 2; c < nch; ++c)
        if ((mask_q >> c) & 1u) after += chunk_escapes(lds128(sw + (uint32_t)(c * kChunkBytes) + 2u * kSlabBytes));
    return pos + qc_mine - after;
}

// The 32 weights of one chunk (BF16 pairs in column order) against x at xs.
template <int MT>
__device__ __forceinline__ void dot32_bf(const uint32_t (&w)[16], uint32_t xs, float (&acc)[MT][4]) {
    uint32_t lo[8], hi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        lo[i] = w[i];
        hi[i] = w[8 + i];
    }
    dot16_bf<MT>(lo, xs, acc);
    dot16_bf<MT>(hi, xs + 32u, acc);
}

// ------------------------------------------------------------------ producer
// The arrival of a range's first piece on its tile's counter, made by the
// producer as soon as the decode warps have stored the piece's partial sums
// (first_done), so that the decode warps never wait for the fence and atomic
// round trip.  The CTAs sharing that tile are still busy with their own
// ranges, so this is rarely the last arrival; if it is, the tile is added up at
// the end of the range (bit 0 of fin_mask).
__device__ __forceinline__ void gemv_first_arrival(const GemmGroup &g, const Piece &pc, volatile int *fin_mask) {
    uint32_t *counter = g.m[pc.member].counters + pc.tile;
    fence_acq_rel_gpu();
    if (arrive_relaxed(counter) == (uint32_t)(pc.count - 1)) {
        fence_acq_rel_gpu();
        *counter = 0u;  // every CTA of the tile has arrived
        atomicOr(const_cast<int *>(fin_mask), 1);  // thread 0 may set bit 1 at the same time
    }
}

template <class C>
__device__ void gemv_sm_producer(const GemmGroup &g, const Piece *pieces, int npieces, const CUtensorMap *tmap,
                                 uint8_t *smem, const GemvBars &b, volatile uint32_t *abort_flag,
                                 volatile int *fin_mask, uint64_t deadline) {
    bool first_pending = npieces > 1 && pieces[0].count > 1;
    uint8_t *hdr = smem + C::kOffHdr;
    const uint64_t stream_policy = policy_evict_first();  // the weights are read once
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
    int gst = 0, gseg = 0;  // weight stages and segment slots issued (one each per segment)
    int hseg = 0;  // headers of the earlier pieces
    for (int k = 0; !stop && k < npieces; ++k) {
        const Piece &pc = pieces[k];
        const GemmParams &p = g.m[pc.member];
        for (int sg = pc.s0; sg < pc.s1; ++sg) {
            const int chunk = sg * kChunksPerSeg;
            const int nch = min(kChunksPerSeg, p.chunks - chunk);
            const int slot = gst % C::kStages;
            if (gst >= C::kStages &&
                !mbar_wait(b.wempty + slot, (uint32_t)(gst / C::kStages - 1) & 1u, deadline)) {
                failed = stop = true;
                break;
            }
            mbar_arrive_expect_tx(b.wfull + slot, (uint32_t)(nch * kChunkBytes));
            bulk_g2s_hint(smem + C::kOffW + slot * C::kWBytes,
                          p.blob + p.off_w + (uint64_t)(pc.tile * p.chunks + chunk) * kChunkBytes,
                          (uint32_t)(nch * kChunkBytes), b.wfull + slot, stream_policy);
            ++gst;
            // the segment's x (no header needed), then its escapes; the one
            // arrival comes last so the phase cannot complete early
            const int sslot = gseg % C::kSegSlots;
            if (gseg >= C::kSegSlots &&
                !mbar_wait(b.sempty + sslot, (uint32_t)(gseg / C::kSegSlots - 1) & 1u, deadline)) {
                failed = stop = true;
                break;
            }
            mbar_expect_tx(b.sfull + sslot, (uint32_t)C::kXbBytes);
            tma_load_2d(smem + C::kOffXb + sslot * C::kXbBytes, tmap, chunk * kChunkK, 0, b.sfull + sslot);
            ++gseg;
            if (!hdr_ready) {
                if (!mbar_wait(b.hdr, 0, deadline)) {
                    mbar_arrive(b.sfull + sslot);  // lets the phase end once x has landed
                    failed = stop = true;
                    break;
                }
                hdr_ready = true;
            }
            const uint4 meta = *reinterpret_cast<const uint4 *>(hdr + (hseg + sg - pc.s0) * kSegHdrBytes + 16);
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
            if (first_pending && mbar_test_wait(b.first_done, 0)) {
                gemv_first_arrival(g, pieces[0], fin_mask);
                first_pending = false;
            }
            if (*abort_flag) {
                stop = true;
                break;
            }
        }
        hseg += pc.s1 - pc.s0;
    }
    // the range's last tile: when the CTAs sharing it have all arrived (they
    // started on it at the beginning of their ranges), pull their slots into
    // L1 now, a few stages before the decoders finish the piece and add them
    if (!failed && !*abort_flag && npieces > 0 && pieces[npieces - 1].count > 1) {
        const Piece &pl = pieces[npieces - 1];
        const GemmParams &p = g.m[pl.member];
        if (load_acquire_gpu(p.counters + pl.tile) == (uint32_t)(pl.count - 1)) {
            const float *base = p.partials + pl.tile * kTileRows;
            for (int sp = 0; sp < pl.count; ++sp)
                if (sp != pl.idx)
                    for (int t = 0; t < p.M; ++t)
#pragma unroll
                        for (int l = 0; l < kTileRows; l += 32)
                            prefetch_l1(base + ((int64_t)sp * p.M + t) * p.Npad + l);
        }
    }
    if (first_pending && !failed && !*abort_flag) {
        if (mbar_wait(b.first_done, 0, deadline))
            gemv_first_arrival(g, pieces[0], fin_mask);
        else
            failed = true;
    }
    mbar_arrive(b.prod_done);  // bit 0 of fin_mask is final
    if (failed) raise_timeout(group_status(g), abort_flag);
    if (*abort_flag) {
        const uint64_t drain_deadline = globaltimer_ns() + 1000000000ull;
        for (int st = max(0, gst - C::kStages); st < gst; ++st)
            mbar_wait(b.wfull + st % C::kStages, (uint32_t)(st / C::kStages) & 1u, drain_deadline);
        for (int sg = max(0, gseg - C::kSegSlots); sg < gseg; ++sg)
            mbar_wait(b.sfull + sg % C::kSegSlots, (uint32_t)(sg / C::kSegSlots) & 1u, drain_deadline);
        mbar_wait(b.hdr, 0, drain_deadline);
    }
}

// ------------------------------------------------------------------ decoders
// One chunk (32 columns) of this thread's row: 32 weights into out0 (columns
// 0-15) and out1 (16-31).  With escapes in the quarter-chunk, run points at
// its first escape byte and moves past the chunk's escapes.
__device__ __forceinline__ void decode_chunk(const Table &T, const uint4 &s0, const uint4 &s1, const uint4 &cd,
                                             bool has_escapes, const uint8_t *&run, uint32_t (&out0)[8],
                                             uint32_t (&out1)[8]) {
    uint32_t E[4];
    if (has_escapes) {
        uint32_t E1[4];
        run += decode_exponents_chunk_esc(T, cd, run, E, E1);
        assemble_half(s0, E, out0);
        assemble_half(s1, E1, out1);
    } else {
        decode_exponents_half(T, cd.x, cd.y, E);
        assemble_half(s0, E, out0);
        decode_exponents_half(T, cd.z, cd.w, E);
        assemble_half(s1, E, out1);
    }
}

// The same chunk as 16 words of BF16 pairs, decoded as if it had no escapes,
// with the escaped exponents patched in afterwards (patch_chunk_escapes): the
// form the tcgen05 kernel uses, whose decode warps are bound by latency
// rather than instruction count.
__device__ __forceinline__ void decode_chunk_patched(const Table &T, const uint4 &s0, const uint4 &s1,
                                                     const uint4 &cd, bool has_escapes, const uint8_t *&run,
                                                     uint32_t (&w)[16]) {
    uint32_t E[4], lo[8], hi[8];
    decode_exponents_half(T, cd.x, cd.y, E);
    assemble_half(s0, E, lo);
    decode_exponents_half(T, cd.z, cd.w, E);
    assemble_half(s1, E, hi);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        w[i] = lo[i];
        w[8 + i] = hi[i];
    }
    if (has_escapes) run += patch_chunk_escapes(cd, run, w);
}

// Per piece: decode and accumulate its segments, then add the four chunk
// groups of each row (j = 1..3 hand their sums to j = 0 through shared
// memory) and write the whole tile's result when the CTA owns the tile, else
// the piece's partial-sum slot.  Only the first and the last piece of a range
// can share their tile with other CTAs; their arrivals are made once at the
// end, and the last arrival adds the tile's slots in slot order.
template <class C>
__device__ void gemv_sm_decode(const GemmGroup &g, const Piece *pieces, int npieces, uint8_t *smem,
                               const GemvBars &b, volatile uint32_t *abort_flag, volatile uint32_t *flag,
                               volatile int *fin_mask, uint64_t deadline) {
    constexpr int MT = C::kMT;
    const int warp = threadIdx.x >> 5;
    const int q = warp & 3;       // rows 32q..32q+31
    const int j = warp >> 2;      // chunks 2j, 2j+1 of each segment
    const int lane = threadIdx.x & 31;
    const int r = 32 * q + lane;  // row in the tile
    const uint8_t *hdr = smem + C::kOffHdr;
    // this thread's S bytes (columns 0-15) of chunk 0 in weight stage 0; the
    // S bytes of columns 16-31 are one slab further on, the codes two
    const uint32_t s_row = smem_u32(smem + C::kOffW) + (uint32_t)(16 * r);
    const uint32_t xb0 = smem_u32(smem + C::kOffXb) + (uint32_t)(2 * j * kChunkK) * 2u;
    float *red = reinterpret_cast<float *>(smem + C::kOffRed);

    // the four j = 0 warps (one per row quarter) meet on an mbarrier pair at
    // most twice per launch; thread 0 runs `lead` in between and writes its
    // result to *flag, which they all read after the meeting
    int meets = 0;
    auto meet = [&](auto lead) -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(b.epi_in);
        if (threadIdx.x == 0) {
            if (mbar_wait(b.epi_in, (uint32_t)meets & 1u, deadline)) {
                *flag = lead() ? 1u : 0u;
                mbar_arrive(b.epi_out);
            } else {
                raise_timeout(group_status(g), abort_flag);
            }
        }
        const bool met = warp_wait(b.epi_out, (uint32_t)meets & 1u, deadline);
        ++meets;
        return met;
    };
    bool ok = warp_wait(b.hdr, 0, deadline);
    int gst = 0;   // stages consumed
    int hseg = 0;  // headers of the earlier pieces
    for (int k = 0; ok && k < npieces; ++k) {
        const Piece &pc = pieces[k];
        const GemmParams &p = g.m[pc.member];
        float acc[MT][4];
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
        for (int sg = pc.s0; sg < pc.s1; ++sg) {
            const int nch = min(kChunksPerSeg, p.chunks - sg * kChunksPerSeg);
            const uint8_t *hp = hdr + (hseg + sg - pc.s0) * kSegHdrBytes;
            const Table T = make_table(*reinterpret_cast<const uint4 *>(hp));
            const uint4 meta = *reinterpret_cast<const uint4 *>(hp + 16);
            const uint32_t mask_q = (meta.w >> (8 * q)) & 0xFFu;
            const int sslot = gst % C::kSegSlots;
            if (!(ok = warp_wait(b.sfull + sslot, (uint32_t)(gst / C::kSegSlots) & 1u, deadline))) break;
            const int slot = gst % C::kStages;
            if (!(ok = warp_wait(b.wfull + slot, (uint32_t)(gst / C::kStages) & 1u, deadline))) break;
            ++gst;
            const int ca = 2 * j;
            const bool va = ca < nch, vb = ca + 1 < nch;  // chunks past a ragged K end are absent
            const uint32_t sa = s_row + (uint32_t)(slot * C::kWBytes + ca * kChunkBytes);
            uint4 a0{}, a1{}, acd{}, b0{}, b1{}, bcd{};
            if (va) {
                a0 = lds128(sa);
                a1 = lds128(sa + kSlabBytes);
                acd = lds128(sa + 2 * kSlabBytes);
            }
            if (vb) {
                b0 = lds128(sa + kChunkBytes);
                b1 = lds128(sa + kChunkBytes + kSlabBytes);
                bcd = lds128(sa + kChunkBytes + 2 * kSlabBytes);
            }
            const uint32_t esc_a = va ? (mask_q >> ca) & 1u : 0u, esc_b = vb ? (mask_q >> (ca + 1)) & 1u : 0u;
            const uint8_t *run = nullptr;
            if (esc_a | esc_b) {
                const uint32_t pos = quarter_chunk_escape_pos(meta, q, j, mask_q, nch, acd, bcd, esc_a, esc_b,
                                                              s_row + (uint32_t)(slot * C::kWBytes));
                if (escapes_staged<C>(seg_escape_total(meta)))
                    run = smem + C::kOffEsc + sslot * C::kEscCap + (meta.x & 15u) + pos;
                else
                    run = p.blob + p.off_esc + meta.x + pos;
            }
            warp_arrive(b.wempty + slot);

            const uint32_t xs = xb0 + (uint32_t)(sslot * C::kXbBytes);
            if (vb && ((esc_a | esc_b) == 0u || MT == 2)) {
                // both chunks present, no escapes: one straight-line block of
                // 32 independent lookup/assembly chains.  With two token rows
                // escaped chunks take it too and have their exponents patched
                // afterwards (as in the tcgen05 kernel); with one, that
                // measured slower (the multiply-adds wait on the patch) and
                // the per-lane table path below serves them
                uint32_t wa[16], wb[16];
                decode_pair_plain(T, a0, a1, acd, b0, b1, bcd, wa, wb);
                if constexpr (MT == 2) {
                    if (esc_a) run += patch_chunk_escapes(acd, run, wa);
                    if (esc_b) run += patch_chunk_escapes(bcd, run, wb);
                }
                dot32_bf<MT>(wa, xs, acc);
                dot32_bf<MT>(wb, xs + (uint32_t)(kChunkK * 2), acc);
            } else {
                if (va) {
                    uint32_t o0[8], o1[8];
                    decode_chunk(T, a0, a1, acd, esc_a != 0u, run, o0, o1);
                    dot16_bf<MT>(o0, xs, acc);
                    dot16_bf<MT>(o1, xs + 32u, acc);
                }
                if (vb) {
                    uint32_t o0[8], o1[8];
                    decode_chunk(T, b0, b1, bcd, esc_b != 0u, run, o0, o1);
                    dot16_bf<MT>(o0, xs + (uint32_t)(kChunkK * 2), acc);
                    dot16_bf<MT>(o1, xs + (uint32_t)(kChunkK * 2) + 32u, acc);
                }
            }
            warp_arrive(b.sempty + sslot);  // done with this segment's x and escapes
        }
        if (!ok) break;
        hseg += pc.s1 - pc.s0;

        // ---- add the four chunk groups of each row in fixed order
        float mine[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) mine[t] = (acc[t][0] + acc[t][1]) + (acc[t][2] + acc[t][3]);
        if (j > 0) {
            // the buffer is free once j = 0 has read the previous piece's sums
            if (k > 0 && !(ok = warp_wait(b.red_empty, (uint32_t)(k - 1) & 1u, deadline))) break;
#pragma unroll
            for (int t = 0; t < MT; ++t) red[((j - 1) * MT + t) * kTileRows + r] = mine[t];
            __syncwarp();
            if (lane == 0) mbar_arrive(b.red);
            continue;
        }
        if (!(ok = warp_wait(b.red, (uint32_t)k & 1u, deadline))) break;
        float total[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t)
            total[t] = ((mine[t] + red[t * kTileRows + r]) + red[(MT + t) * kTileRows + r]) +
                       red[(2 * MT + t) * kTileRows + r];
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
        uint32_t *counter = p.counters + pc.tile;
        if (k == npieces - 1) {
            // the range's last piece: the CTAs sharing its tile normally
            // arrived long ago (at the start of their ranges); then add their
            // slots to this piece's sums, still in registers, in slot order
            ok = meet([&] { return load_acquire_gpu(counter) == (uint32_t)(pc.count - 1); });
            if (!ok) break;
            if (*flag) {
                const float *src = p.partials + (n < p.N ? n : pc.tile * kTileRows);
                const int64_t stride = (int64_t)p.M * p.Npad;
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    if (t >= p.M) continue;
                    float s = 0.0f;
                    // through L1: the acquire above showed the slots complete
                    // (and the producer may have prefetched them)
                    for (int sp = 0; sp < pc.count; ++sp)
                        s += sp == pc.idx ? total[t] : __ldca(src + (int64_t)t * p.Npad + (int64_t)sp * stride);
                    if (p.y != nullptr && n < p.N) p.y[(int64_t)t * p.N + n] = bf16_bits_rn(s);
                    if (p.amax != nullptr) argmax_warp(p.amax + t, n < p.N ? argmax_key(s, (uint32_t)n) : 0ull);
                }
                if (threadIdx.x == 0) *counter = 0u;  // every CTA of the tile has arrived
                continue;
            }
        }
#pragma unroll
        for (int t = 0; t < MT; ++t)
            if (t < p.M) __stcg(p.partials + ((int64_t)pc.idx * p.M + t) * p.Npad + n, total[t]);
        if (k < npieces - 1) {
            // the first piece: the producer arrives for it once all four warps
            // have stored their rows (the mbarrier orders the stores first)
            __syncwarp();
            if (lane == 0) mbar_arrive(b.first_done);
            continue;
        }
        // the last piece, others still missing: arrive now
        ok = meet([&] {
            fence_acq_rel_gpu();
            const bool last = arrive_relaxed(counter) == (uint32_t)(pc.count - 1);
            if (last) {
                fence_acq_rel_gpu();
                *counter = 0u;
                atomicOr(const_cast<int *>(fin_mask), 2);
            }
            return last;
        });
        if (!ok) break;
    }
    if (!ok) {
        if (lane == 0) raise_timeout(group_status(g), abort_flag);
        return;
    }
    if (j > 0) return;

    // ---- tiles this CTA completed as the last arrival, added up from memory
    // in slot order (the producer's word on the first piece comes first)
    if (!warp_wait(b.prod_done, 0, deadline)) {
        if (lane == 0) raise_timeout(group_status(g), abort_flag);
        return;
    }
    const int mask = *fin_mask;
    for (int e = 0; e < 2; ++e) {
        if (!((mask >> e) & 1)) continue;
        const Piece &pc = pieces[e == 0 ? 0 : npieces - 1];
        const GemmParams &p = g.m[pc.member];
        const int64_t n = pc.tile * kTileRows + r;
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            if (t >= p.M) continue;
            const float *src = p.partials + (int64_t)t * p.Npad + (n < p.N ? n : pc.tile * kTileRows);
            const int64_t stride = (int64_t)p.M * p.Npad;
            float s = 0.0f;
            for (int sp = 0; sp < pc.count; sp += 8) {
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
    }
}

// ------------------------------------------------------------------ kernel
template <int MT>
__global__ void __launch_bounds__(GemvSmCfg<MT>::kThreads, 1)
    w12_gemv_sm_kernel(const __grid_constant__ GemmGroup grp, const __grid_constant__ CUtensorMap tmap_x) {
    using C = GemvSmCfg<MT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBars);
    GemvBars b;
    b.wfull = bars;
    b.wempty = b.wfull + C::kStages;
    b.sfull = b.wempty + C::kStages;
    b.sempty = b.sfull + C::kSegSlots;
    b.hdr = b.sempty + C::kSegSlots;
    b.red = b.hdr + 1;
    b.red_empty = b.red + 1;
    b.epi_in = b.red_empty + 1;
    b.epi_out = b.epi_in + 1;
    b.first_done = b.epi_out + 1;
    b.prod_done = b.first_done + 1;
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile uint32_t *abort_flag = misc + 1;
    volatile uint32_t *npieces = misc + 2;
    volatile uint32_t *flag = misc + 4;  // thread 0's word to the j = 0 warps
    volatile int *fin_mask = reinterpret_cast<volatile int *>(misc + 5);  // tiles to add up at the end
    Piece *pieces = reinterpret_cast<Piece *>(smem + C::kOffPieces);

    const int warp = threadIdx.x >> 5;
    const uint64_t deadline = globaltimer_ns() + grp.m[0].timeout_ns;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(b.wfull + i, 1);
            mbar_init(b.wempty + i, C::kDecWarps);
        }
        for (int i = 0; i < C::kSegSlots; ++i) {
            mbar_init(b.sfull + i, 1);
            mbar_init(b.sempty + i, C::kDecWarps);
        }
        mbar_init(b.hdr, 1);
        mbar_init(b.red, 12);
        mbar_init(b.red_empty, 4);
        mbar_init(b.epi_in, 4);
        mbar_init(b.epi_out, 1);
        mbar_init(b.first_done, 4);
        mbar_init(b.prod_done, 1);
        *flag = 0u;
        *fin_mask = 0;
        *abort_flag = 0u;
        // this CTA's pieces (the planner keeps them within kMaxPieces)
        CtaWork w = cta_work(grp);
        uint32_t n = 0;
        while (n < C::kMaxPieces && next_piece(grp, w, pieces[n])) ++n;
        *npieces = n;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) pdl_launch_dependents();
    const int np = (int)*npieces;
    if (warp == C::kDecWarps && (threadIdx.x & 31) == 0) prefetch_pieces<kChunkBytes, true>(grp, pieces, np);
    pdl_wait();
    if (warp == C::kDecWarps) {
        if ((threadIdx.x & 31) == 0) gemv_sm_producer<C>(grp, pieces, np, &tmap_x, smem, b, abort_flag, fin_mask, deadline);
    } else {
        gemv_sm_decode<C>(grp, pieces, np, smem, b, abort_flag, flag, fin_mask, deadline);
    }
}

}  // namespace dev
}  // namespace w12
