// W12 decode-GEMM on tcgen05 tensor cores with one CTA per SM (sm_103a): y =
// x . W^T for 3..32 tokens, W streamed from HBM in W12 form and decoded in
// registers ("decoded inside the GEMM registers", "SpecPilot: an agent
// doubled speculative decoding speed, and the 10.87x needs context", §The
// mechanisms it found; bit-exact weights, "StargazerX0/SpecPilot", §What it
// is; 12 instead of 16 bits cut the traffic of a memory-bound decode by a
// quarter, same section of the first page).
//
// The arithmetic is that of gemm_tc.cuh (swap-AB: a decoded 128-row tile of W
// is the A operand, x the B operand with N = 16 or 32 tokens, fp32
// accumulators in TMEM); what differs is how an SM's warps share the work.
// Several small CTAs per SM, each with its own short rings and handshakes,
// leave the SM's last stretch to whichever CTA the scheduler placed second.
// Here one CTA owns the SM, a weight stage is a whole 256-column segment
// (48 KB), sixteen warps decode it together, and the CTA walks a contiguous
// stream-K range of (tile, segment) units, so one wave covers the launch
// with equal work per SM whatever the tile count.
//
// Warp roles (704 threads):
//   warps 0-15  decode: warp w handles rows 32q..32q+31 (q = w mod 4, the TMEM
//               lanes its warp may touch) and chunks 2j, 2j+1 of each segment
//               (j = w / 4); per stage a thread reads its row's S bytes and
//               codes of its two chunks from SMEM, decodes 64 weights,
//               patches escapes and stores them as 32 columns of BF16 pairs
//               into a TMEM A slot (one slot per segment, 128 columns);
//   warp 16     producer: cp.async.bulk for the segment headers and each
//               weight stage; per segment cp.async.bulk.tensor for the x tile
//               (four 64-column boxes, 128-byte swizzle) and cp.async.bulk for
//               the escape bytes;
//   warp 17     allocates TMEM (all 512 columns); one lane issues the 16
//               MMAs of a segment (K = 16 each) into the piece's accumulator
//               and tcgen05.commit;
//   warps 18-21 epilogue: one warp per TMEM lane quarter drains a finished
//               piece's accumulator (two accumulators alternate, so the MMAs
//               of the next piece do not wait) and writes y, or the piece's
//               partial-sum slot when the tile is shared with other CTAs.
// A range's first and last pieces may share their tile; their arrivals are
// made once at the end and the last arrival adds the tile's slots in slot
// order, so results repeat run to run.  Every wait is bounded: on expiry the
// kernel records W12_ERR_TIMEOUT, lets copies land and MMAs finish, frees
// TMEM and returns.
#pragma once

#include "gemv_sm.cuh"

namespace w12 {
namespace dev {

template <int NTOK>
struct TcSmCfg {
    static constexpr int kNtok = NTOK;
    static constexpr int kDecWarps = 16;
    static constexpr int kProdWarp = 16;
    static constexpr int kMmaWarp = 17;
    static constexpr int kEpiWarp0 = 18;  // warps 18..21 cover lane quarters 2, 3, 0, 1
    static constexpr int kEpiWarps = 4;
    static constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;
    static constexpr int kStages = 3;                            // weight ring: one segment per stage
    static constexpr int kWBytes = kChunksPerSeg * kChunkBytes;  // 48 KB
    static constexpr int kXBoxBytes = NTOK * 128;                // 64 columns x NTOK tokens
    static constexpr int kXBytes = 4 * kXBoxBytes;               // x tile of one segment
    static constexpr int kSegSlots = NTOK == 32 ? 3 : 4;         // x + escapes, one segment each
    static constexpr int kEscCap = 2048;
    static constexpr int kASlots = 3;                            // TMEM A slots, one segment each
    static constexpr int kMaxSegs = 192;                         // units (segments) of one CTA
    static constexpr int kMaxPieces = 64;                        // tiles one CTA's range meets
    static constexpr int kTmemCols = 512;
    static constexpr int kDCol = 0;                              // accumulators at columns 0 and 32
    static constexpr int kACol = 64;                             // A slot s at 64 + 128 s
    static constexpr int kOffX = 0;                              // 1024-aligned (swizzle atoms)
    static constexpr int kOffW = kOffX + kSegSlots * kXBytes;
    static constexpr int kOffEsc = kOffW + kStages * kWBytes;
    static constexpr int kOffHdr = kOffEsc + kSegSlots * kEscCap;
    static constexpr int kOffBars = kOffHdr + kMaxSegs * kSegHdrBytes;
    // wfull[S], wempty[S], sfull[X], sempty[X], afull[A], aempty[A], dfull[2],
    // dempty[2], hdr, drain, epi_in, epi_out
    static constexpr int kNumBars = 2 * kStages + 2 * kSegSlots + 2 * kASlots + 4 + 4;
    static constexpr int kOffMisc = kOffBars + kNumBars * 8;
    static constexpr int kOffPieces = kOffMisc + 64;
    static constexpr int kSmemBytes = kOffPieces + kMaxPieces * (int)sizeof(Piece) + 1024;  // + alignment slack
    static_assert(NTOK == 16 || NTOK == 32, "token tile is 16 or 32");
    static_assert(kXBoxBytes % 1024 == 0, "x boxes must stay 1024-byte aligned for the 128-byte swizzle");
    static_assert(kOffW % 128 == 0 && kOffEsc % 16 == 0 && kOffHdr % 16 == 0, "copy destinations aligned");
    static_assert(kACol + kASlots * 128 <= kTmemCols && kDCol + 64 <= kACol, "TMEM columns");
    static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM must fit");
};

struct TcSmBars {
    uint64_t *wfull, *wempty, *sfull, *sempty, *afull, *aempty, *dfull, *dempty, *hdr, *drain, *epi_in, *epi_out;
};

// ------------------------------------------------------------------ producer
template <class C>
__device__ void tcsm_producer(const GemmGroup &g, const Piece *pieces, int npieces, const CUtensorMap *tmap,
                              uint8_t *smem, const TcSmBars &b, volatile uint32_t *abort_flag, uint64_t deadline) {
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
    int gw = 0, gx = 0;  // weight stages and x slots issued (one each per segment)
    int hseg = 0;        // headers of the earlier pieces
    for (int k = 0; !stop && k < npieces; ++k) {
        const Piece &pc = pieces[k];
        const GemmParams &p = g.m[pc.member];
        for (int sg = pc.s0; sg < pc.s1; ++sg) {
            const int chunk = sg * kChunksPerSeg;
            const int nch = min(kChunksPerSeg, p.chunks - chunk);
            const int wslot = gw % C::kStages;
            if (gw >= C::kStages && !mbar_wait(b.wempty + wslot, (uint32_t)(gw / C::kStages - 1) & 1u, deadline)) {
                failed = stop = true;
                break;
            }
            mbar_arrive_expect_tx(b.wfull + wslot, (uint32_t)(nch * kChunkBytes));
            bulk_g2s(smem + C::kOffW + wslot * C::kWBytes,
                     p.blob + p.off_w + (uint64_t)(pc.tile * p.chunks + chunk) * kChunkBytes,
                     (uint32_t)(nch * kChunkBytes), b.wfull + wslot);
            ++gw;
            // the segment's x tile (no header needed), then its escapes; the
            // one arrival comes last so the phase cannot complete early
            const int xslot = gx % C::kSegSlots;
            if (gx >= C::kSegSlots &&
                !mbar_wait(b.sempty + xslot, (uint32_t)(gx / C::kSegSlots - 1) & 1u, deadline)) {
                failed = stop = true;
                break;
            }
            mbar_expect_tx(b.sfull + xslot, (uint32_t)C::kXBytes);
            uint8_t *xs = smem + C::kOffX + xslot * C::kXBytes;
#pragma unroll
            for (int bx = 0; bx < 4; ++bx)
                tma_load_2d(xs + bx * C::kXBoxBytes, tmap, chunk * kChunkK + bx * 64, 0, b.sfull + xslot);
            ++gx;
            if (!hdr_ready) {
                if (!mbar_wait(b.hdr, 0, deadline)) {
                    mbar_arrive(b.sfull + xslot);  // lets the phase end once x has landed
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
                mbar_expect_tx(b.sfull + xslot, ebytes);
                bulk_g2s(smem + C::kOffEsc + xslot * C::kEscCap, p.blob + p.off_esc + src0, ebytes,
                         b.sfull + xslot);
            }
            mbar_arrive(b.sfull + xslot);
            if (*abort_flag) {
                stop = true;
                break;
            }
        }
        hseg += pc.s1 - pc.s0;
    }
    if (failed) raise_timeout(group_status(g), abort_flag);
    if (*abort_flag) {
        // let every copy still in flight land before the CTA can exit
        const uint64_t drain_deadline = globaltimer_ns() + 1000000000ull;
        for (int st = max(0, gw - C::kStages); st < gw; ++st)
            mbar_wait(b.wfull + st % C::kStages, (uint32_t)(st / C::kStages) & 1u, drain_deadline);
        for (int sx = max(0, gx - C::kSegSlots); sx < gx; ++sx)
            mbar_wait(b.sfull + sx % C::kSegSlots, (uint32_t)(sx / C::kSegSlots) & 1u, drain_deadline);
        mbar_wait(b.hdr, 0, drain_deadline);
    }
}

// ------------------------------------------------------------------ MMA issuer
// Segment gs of the CTA's range: 2 x nch MMAs of K = 16.  A: TMEM slot
// gs mod 3, columns 8 kb .. 8 kb + 7 for k-block kb (the decoders store a
// chunk's 32 columns as 16 consecutive columns of BF16 pairs).  B: the x
// tile, four 128-byte-swizzled 64-column boxes, K-major, 8-row atoms of 1024
// bytes; k-block kb starts 32 (kb mod 4) bytes into box kb / 4.
template <class C>
__device__ void tcsm_mma(const GemmGroup &g, const Piece *pieces, int npieces, uint8_t *smem, const TcSmBars &b,
                         volatile uint32_t *abort_flag, uint32_t tmem_base, uint64_t deadline) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, C::kNtok);
    bool failed = false;
    int gs = 0;
    for (int k = 0; !failed && k < npieces; ++k) {
        const Piece &pc = pieces[k];
        const GemmParams &p = g.m[pc.member];
        const int dbuf = k & 1;
        // the accumulator is free once the epilogue has read piece k - 2
        if (k >= 2 && !mbar_wait(b.dempty + dbuf, (uint32_t)((k >> 1) - 1) & 1u, deadline)) {
            failed = true;
            break;
        }
        tc_fence_after();
        const uint32_t d_taddr = tmem_base + (uint32_t)(C::kDCol + 32 * dbuf);
        for (int sg = pc.s0; sg < pc.s1; ++sg, ++gs) {
            const int nch = min(kChunksPerSeg, p.chunks - sg * kChunksPerSeg);
            const int xslot = gs % C::kSegSlots, aslot = gs % C::kASlots;
            if (!mbar_wait(b.sfull + xslot, (uint32_t)(gs / C::kSegSlots) & 1u, deadline) ||
                !mbar_wait(b.afull + aslot, (uint32_t)(gs / C::kASlots) & 1u, deadline)) {
                failed = true;
                break;
            }
            tc_fence_after();
            const uint32_t xs = smem_u32(smem + C::kOffX + xslot * C::kXBytes);
            const uint32_t a_taddr = tmem_base + (uint32_t)(C::kACol + 128 * aslot);
            for (int kb = 0; kb < 2 * nch; ++kb) {
                const uint64_t bdesc =
                    smem_desc(xs + (uint32_t)(kb >> 2) * C::kXBoxBytes + (uint32_t)(kb & 3) * 32u, 16u, 1024u, 2u);
                mma_tmem_a(d_taddr, a_taddr + (uint32_t)(8 * kb), bdesc, idesc, (sg > pc.s0 || kb > 0) ? 1u : 0u);
            }
            mma_commit(b.aempty + aslot);
            mma_commit(b.sempty + xslot);
            if (*abort_flag) {
                failed = true;
                break;
            }
        }
        if (!failed) mma_commit(b.dfull + dbuf);
    }
    if (failed) raise_timeout(group_status(g), abort_flag);
    // before TMEM can be freed every issued MMA must have completed
    mma_commit(b.drain);
    mbar_wait(b.drain, 0, globaltimer_ns() + 1000000000ull);
}

// ------------------------------------------------------------------ decoders
// Escapes of quarter-chunk c of the stage in weight slot `slot` (this warp's
// rows): the warp total, from the chunk's codes.
__device__ __forceinline__ uint32_t stage_chunk_escapes(uint32_t s_row_slot, int c) {
    return chunk_escapes(lds128(s_row_slot + (uint32_t)(c * kChunkBytes) + 2u * kSlabBytes));
}

// Decode one chunk of this thread's row and store its 32 weights as 16 TMEM
// columns of BF16 pairs (column c: weights 2c, 2c + 1) at taddr.
__device__ __forceinline__ void decode_chunk_to_tmem(const Table &T, const uint4 &s0, const uint4 &s1,
                                                     const uint4 &cd, bool has_escapes, const uint8_t *&run,
                                                     uint32_t taddr) {
    uint32_t lo[8], hi[8], v[16];
    decode_chunk(T, s0, s1, cd, has_escapes, run, lo, hi);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[i] = lo[i];
        v[8 + i] = hi[i];
    }
    tmem_st16(taddr, v);
}

template <class C>
__device__ void tcsm_decode(const GemmGroup &g, const Piece *pieces, int npieces, uint8_t *smem, const TcSmBars &b,
                            volatile uint32_t *abort_flag, uint32_t tmem_base, uint64_t deadline) {
    const int warp = threadIdx.x >> 5;
    const int q = warp & 3;       // TMEM lane quarter = rows 32q..32q+31
    const int j = warp >> 2;      // chunks 2j, 2j+1 of each segment
    const int lane = threadIdx.x & 31;
    const int r = 32 * q + lane;  // row in the tile
    const uint8_t *hdr = smem + C::kOffHdr;
    const uint32_t s_row = smem_u32(smem + C::kOffW) + (uint32_t)(16 * r);
    const uint32_t a_lane = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(C::kACol + 32 * j);

    bool ok = warp_wait(b.hdr, 0, deadline);
    int gs = 0;     // segments of the range so far
    int hseg = 0;   // headers of the earlier pieces
    int pend = -1;  // A slot whose stores still await their handshake
    for (int k = 0; ok && k < npieces; ++k) {
        const Piece &pc = pieces[k];
        const GemmParams &p = g.m[pc.member];
        for (int sg = pc.s0; sg < pc.s1; ++sg, ++gs) {
            const int nch = min(kChunksPerSeg, p.chunks - sg * kChunksPerSeg);
            const uint8_t *hp = hdr + (hseg + sg - pc.s0) * kSegHdrBytes;
            const Table T = make_table(*reinterpret_cast<const uint4 *>(hp));
            const uint4 meta = *reinterpret_cast<const uint4 *>(hp + 16);
            const uint32_t mask_q = (meta.w >> (8 * q)) & 0xFFu;
            const int xslot = gs % C::kSegSlots, wslot = gs % C::kStages;
            if (!(ok = warp_wait(b.wfull + wslot, (uint32_t)(gs / C::kStages) & 1u, deadline))) break;
            const int ca = 2 * j;
            const bool va = ca < nch, vb = ca + 1 < nch;  // chunks past a ragged K end are absent
            const uint32_t sw = s_row + (uint32_t)(wslot * C::kWBytes);
            const uint32_t sa = sw + (uint32_t)(ca * kChunkBytes);
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
            // every decoder waits for the segment slot before it releases it:
            // an early release could count toward the slot's previous use
            bool have_slot = false;
            if (esc_a | esc_b) {
                // the quarter's escapes run chunk by chunk; find where chunk 2j's
                // start from whichever end of the quarter has fewer chunks to
                // count: the earlier chunks (j < 2), or the quarter's total
                // minus this and the later chunks (j >= 2)
                const uint32_t qc0 = meta.y & 0xFFFFu, qc1 = meta.y >> 16, qc2 = meta.z & 0xFFFFu;
                const uint32_t qc_mine = ((q < 2 ? meta.y : meta.z) >> (16 * (q & 1))) & 0xFFFFu;
                uint32_t pos = (q > 0 ? qc0 : 0u) + (q > 1 ? qc1 : 0u) + (q > 2 ? qc2 : 0u);
                if (j < 2) {
                    for (int c = 0; c < ca; ++c)
                        if ((mask_q >> c) & 1u) pos += stage_chunk_escapes(sw, c);
                } else {
                    uint32_t after = 0;
                    if (esc_a) after += chunk_escapes(acd);
                    if (esc_b) after += chunk_escapes(bcd);
                    for (int c = ca + 2; c < nch; ++c)
                        if ((mask_q >> c) & 1u) after += stage_chunk_escapes(sw, c);
                    pos += qc_mine - after;
                }
                if (!(ok = warp_wait(b.sfull + xslot, (uint32_t)(gs / C::kSegSlots) & 1u, deadline))) break;
                have_slot = true;
                if (escapes_staged<C>(seg_escape_total(meta)))
                    run = smem + C::kOffEsc + xslot * C::kEscCap + (meta.x & 15u) + pos;
                else
                    run = p.blob + p.off_esc + meta.x + pos;
            }
            warp_arrive(b.wempty + wslot);  // this warp is done with the stage's bytes

            // the previous segment's stores: wait for them, then hand the slot
            // to the MMA warp (one segment late, so that the store latency
            // overlaps this segment's loads)
            if (pend >= 0) {
                tmem_wait_st();
                tc_fence_before();
                warp_arrive(b.afull + pend);
                pend = -1;
            }
            const int aslot = gs % C::kASlots;
            if (gs >= C::kASlots &&
                !(ok = warp_wait(b.aempty + aslot, (uint32_t)(gs / C::kASlots - 1) & 1u, deadline)))
                break;
            tc_fence_after();
            // each chunk goes to TMEM as soon as it is decoded: 16 columns of
            // BF16 pairs, the chunk's 32 weights in column order
            const uint32_t ta = a_lane + (uint32_t)(128 * aslot);
            if (va) decode_chunk_to_tmem(T, a0, a1, acd, esc_a != 0u, run, ta);
            if (vb) decode_chunk_to_tmem(T, b0, b1, bcd, esc_b != 0u, run, ta + 16u);
            if (!have_slot && !(ok = warp_wait(b.sfull + xslot, (uint32_t)(gs / C::kSegSlots) & 1u, deadline))) {
                pend = aslot;
                break;
            }
            warp_arrive(b.sempty + xslot);  // done with this segment's escapes
            pend = aslot;
            if (*abort_flag) {
                ok = false;
                break;
            }
        }
        hseg += pc.s1 - pc.s0;
    }
    if (pend >= 0) {
        tmem_wait_st();
        tc_fence_before();
        if (ok) warp_arrive(b.afull + pend);
    }
    if (!ok && lane == 0) raise_timeout(group_status(g), abort_flag);
}

// ------------------------------------------------------------------ epilogue
// One warp per TMEM lane quarter: for each piece, wait for its accumulator,
// read this quarter's 32 rows x NTOK tokens, release the accumulator, then
// store y (the CTA owns the tile) or the piece's partial-sum slot.  After the
// last piece, the shared first and last pieces arrive on their tiles'
// counters, and the last arrival of a tile adds its slots in slot order.
template <class C>
__device__ void tcsm_epilogue(const GemmGroup &g, const Piece *pieces, int npieces, const TcSmBars &b,
                              volatile uint32_t *abort_flag, volatile uint32_t *last_flags, uint32_t tmem_base,
                              uint64_t deadline) {
    constexpr int NT = C::kNtok;
    const int warp = threadIdx.x >> 5;
    const int q = warp & 3;
    const int lane = threadIdx.x & 31;
    const int r = 32 * q + lane;
    const uint32_t d_lane = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)C::kDCol;
    bool ok = true;
    for (int k = 0; k < npieces; ++k) {
        const Piece &pc = pieces[k];
        const GemmParams &p = g.m[pc.member];
        const int dbuf = k & 1;
        if (!(ok = warp_wait(b.dfull + dbuf, (uint32_t)(k >> 1) & 1u, deadline))) break;
        tc_fence_after();
        float acc[NT];
        {
            uint32_t v[16];
#pragma unroll
            for (int h = 0; h < NT / 16; ++h) {
                tmem_ld16(d_lane + (uint32_t)(32 * dbuf + 16 * h), v);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 16; ++t) acc[16 * h + t] = __uint_as_float(v[t]);
            }
        }
        tc_fence_before();
        warp_arrive(b.dempty + dbuf);
        const int64_t n = pc.tile * kTileRows + r;
        if (pc.count == 1) {
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                if (t < p.M) {
                    if (p.y != nullptr && n < p.N) p.y[(int64_t)t * p.N + n] = bf16_bits_rn(acc[t]);
                    if (p.amax != nullptr) argmax_warp(p.amax + t, n < p.N ? argmax_key(acc[t], (uint32_t)n) : 0ull);
                }
            }
            continue;
        }
#pragma unroll
        for (int t = 0; t < NT; ++t)
            if (t < p.M) __stcg(p.partials + ((int64_t)pc.idx * p.M + t) * p.Npad + n, acc[t]);
    }
    if (!ok) {
        if (lane == 0) raise_timeout(group_status(g), abort_flag);
        return;
    }
    // the pieces that share their tile: the first and the last (one when equal)
    const int ka = 0, kb = npieces - 1;
    const bool sa = npieces > 0 && pieces[ka].count > 1;
    const bool sb = kb > ka && pieces[kb].count > 1;
    if (!(sa || sb)) return;

    // split-K arrivals, once at the end: the mbarrier arrive/wait pair orders
    // the four warps' partial stores before one thread's release fence, which
    // with the increments after it publishes them
    __syncwarp();
    const bool leader = warp == C::kEpiWarp0 && lane == 0;
    if (lane == 0) mbar_arrive(b.epi_in);
    if (leader) {
        if (mbar_wait(b.epi_in, 0, deadline)) {
            fence_acq_rel_gpu();
            uint32_t oa = 0, ob = 0;
            if (sa) oa = arrive_relaxed(g.m[pieces[ka].member].counters + pieces[ka].tile);
            if (sb) ob = arrive_relaxed(g.m[pieces[kb].member].counters + pieces[kb].tile);
            const bool la = sa && oa == (uint32_t)(pieces[ka].count - 1);
            const bool lb = sb && ob == (uint32_t)(pieces[kb].count - 1);
            last_flags[0] = la ? 1u : 0u;
            last_flags[1] = lb ? 1u : 0u;
            if (la || lb) fence_acq_rel_gpu();
            mbar_arrive(b.epi_out);
        } else {
            raise_timeout(group_status(g), abort_flag);
        }
    }
    if (!warp_wait(b.epi_out, 0, deadline)) {
        if (lane == 0) raise_timeout(group_status(g), abort_flag);
        return;
    }
    for (int e = 0; e < 2; ++e) {
        if (last_flags[e] == 0) continue;
        const Piece &pc = pieces[e == 0 ? ka : kb];
        const GemmParams &p = g.m[pc.member];
        const int64_t n = pc.tile * kTileRows + r;
        const int64_t stride = (int64_t)p.M * p.Npad;
        for (int t = 0; t < p.M; ++t) {
            const float *src = p.partials + (int64_t)t * p.Npad + (n < p.N ? n : pc.tile * kTileRows);
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
        if (leader) p.counters[pc.tile] = 0u;  // ready for the next call
    }
}

// ------------------------------------------------------------------ kernel
template <int NTOK>
__global__ void __launch_bounds__(TcSmCfg<NTOK>::kThreads, 1)
    w12_gemm_tc_sm_kernel(const __grid_constant__ GemmGroup grp, const __grid_constant__ CUtensorMap tmap_x) {
    using C = TcSmCfg<NTOK>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBars);
    TcSmBars b;
    b.wfull = bars;
    b.wempty = b.wfull + C::kStages;
    b.sfull = b.wempty + C::kStages;
    b.sempty = b.sfull + C::kSegSlots;
    b.afull = b.sempty + C::kSegSlots;
    b.aempty = b.afull + C::kASlots;
    b.dfull = b.aempty + C::kASlots;
    b.dempty = b.dfull + 2;
    b.hdr = b.dempty + 2;
    b.drain = b.hdr + 1;
    b.epi_in = b.drain + 1;
    b.epi_out = b.epi_in + 1;
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    uint32_t *tmem_slot = misc;
    volatile uint32_t *abort_flag = misc + 1;
    volatile uint32_t *npieces = misc + 2;
    volatile uint32_t *last_flags = misc + 4;  // [2]
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
            mbar_init(b.sempty + i, C::kDecWarps + 1);  // decoders done with the escapes + MMAs done with x
        }
        for (int i = 0; i < C::kASlots; ++i) {
            mbar_init(b.afull + i, C::kDecWarps);
            mbar_init(b.aempty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(b.dfull + i, 1);
            mbar_init(b.dempty + i, C::kEpiWarps);
        }
        mbar_init(b.hdr, 1);
        mbar_init(b.drain, 1);
        mbar_init(b.epi_in, C::kEpiWarps);
        mbar_init(b.epi_out, 1);
        *abort_flag = 0u;
        last_flags[0] = last_flags[1] = 0u;
        // this CTA's pieces (the planner keeps them within kMaxPieces)
        CtaWork w = cta_work(grp);
        uint32_t n = 0;
        while (n < C::kMaxPieces && next_piece(grp, w, pieces[n])) ++n;
        *npieces = n;
        fence_mbar_init();
    }
    if (warp == C::kMmaWarp) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0) pdl_launch_dependents();
    const int np = (int)*npieces;
    if (warp == C::kProdWarp && (threadIdx.x & 31) == 0) prefetch_pieces<kChunkBytes, true>(grp, pieces, np);
    pdl_wait();

    if (warp == C::kProdWarp) {
        if ((threadIdx.x & 31) == 0) tcsm_producer<C>(grp, pieces, np, &tmap_x, smem, b, abort_flag, deadline);
    } else if (warp == C::kMmaWarp) {
        if ((threadIdx.x & 31) == 0) tcsm_mma<C>(grp, pieces, np, smem, b, abort_flag, tmem_base, deadline);
        __syncwarp();
    } else if (warp >= C::kEpiWarp0) {
        tcsm_epilogue<C>(grp, pieces, np, b, abort_flag, last_flags, tmem_base, deadline);
    } else {
        tcsm_decode<C>(grp, pieces, np, smem, b, abort_flag, tmem_base, deadline);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::kMmaWarp) tmem_dealloc(tmem_base, C::kTmemCols);
}

}  // namespace dev
}  // namespace w12
