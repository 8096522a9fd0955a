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
// Warp roles (736 threads):
//   warps 0-15  decode: warp w handles rows 32q..32q+31 (q = w mod 4, the TMEM
//               lanes its warp may touch) and chunks 2j, 2j+1 of each segment
//               (j = w / 4); per stage a thread reads its row's S bytes and
//               codes of its two chunks from SMEM, decodes 64 weights,
//               patches escapes and stores them as 32 columns of BF16 pairs
//               into a TMEM A slot (one slot per segment, 128 columns);
//   warp 16     weight producer: cp.async.bulk for the segment headers, each
//               weight stage and each segment's escape bytes (their own ring,
//               one slot deeper than the weight ring, so the weight stage is
//               free as soon as the decoders have read it and an escape slot
//               is known free when the following weight stage is);
//   warp 17     allocates TMEM (all 512 columns); one lane issues the 16
//               MMAs of a segment (K = 16 each) into the piece's accumulator
//               and tcgen05.commit;
//   warps 18-21 epilogue: one warp per TMEM lane quarter drains a finished
//               piece's accumulator (two accumulators alternate, so the MMAs
//               of the next piece do not wait) and writes y, or the piece's
//               partial-sum slot when the tile is shared with other CTAs;
//   warp 22     x loader: per segment cp.async.bulk.tensor for the x tile
//               (four 64-column boxes, 128-byte swizzle) into a ring of its
//               own, whose slots the MMAs free; kept apart from the weight
//               producer so that no weight stage waits for an MMA.
// A range's first and last pieces may share their tile; their arrivals are
// made once at the end and the last arrival adds the tile's slots in slot
// order, so results repeat run to run.  Every wait is bounded: on expiry the
// kernel records W12_ERR_TIMEOUT, lets copies land and MMAs finish, frees
// TMEM and returns.
#pragma once

#include "gemv_sm.cuh"

namespace w12 {
namespace dev {

template <int NTOK, bool Q8 = false>
struct TcSmCfg {
    static constexpr int kNtok = NTOK;
    static constexpr bool kQ8 = Q8;                              // weights: the Q8 copy instead of W12
    static constexpr int kChunkB = Q8 ? q8::kChunkBytes : kChunkBytes;
    static constexpr int kDecWarps = 16;
    static constexpr int kProdWarp = 16;
    static constexpr int kMmaWarp = 17;
    static constexpr int kEpiWarp0 = 18;  // warps 18..21 cover lane quarters 2, 3, 0, 1
    static constexpr int kEpiWarps = 4;
    static constexpr int kXWarp = 22;
    static constexpr int kThreads = (kXWarp + 1) * 32;
    static constexpr int kFinishThreads = (kDecWarps + kEpiWarps) * 32;  // share a split-K finish
    // weight ring: one segment per stage (48 KB of W12, three deep; 32 KB of
    // Q8, four deep)
    static constexpr int kStages = Q8 ? 4 : 3;
    static constexpr int kWBytes = kChunksPerSeg * kChunkB;
    static constexpr int kXBoxBytes = NTOK * 128;                // 64 columns x NTOK tokens
    static constexpr int kXBytes = 4 * kXBoxBytes;               // x tile of one segment
    static constexpr int kXSlots = 4;                            // x ring
    static constexpr int kESlots = Q8 ? 1 : kStages + 1;         // escape-byte ring, one deeper than the weights
    static constexpr int kEscCap = 2048;
    static constexpr int kASlots = 3;                            // TMEM A slots, one segment each
    static constexpr int kMaxSegs = 192;                         // units (segments) of one CTA
    static constexpr int kMaxPieces = 64;                        // tiles one CTA's range meets
    static constexpr int kTmemCols = 512;
    static constexpr int kDCol = 0;                              // accumulators at columns 0 and 32
    static constexpr int kACol = 64;                             // A slot s at 64 + 128 s
    static constexpr int kOffX = 0;                              // 1024-aligned (swizzle atoms)
    static constexpr int kOffW = kOffX + kXSlots * kXBytes;
    static constexpr int kOffEsc = kOffW + kStages * kWBytes;
    static constexpr int kOffHdr = kOffEsc + kESlots * kEscCap;
    static constexpr int kOffBars = kOffHdr + kMaxSegs * kSegHdrBytes;
    // wfull[S], wempty[S], efull[E], xfull[X], xempty[X], afull[A],
    // aempty[A], dfull[2], dempty[2], hdr, drain, epi_in, epi_out, fin
    static constexpr int kNumBars = 2 * kStages + kESlots + 2 * kXSlots + 2 * kASlots + 4 + 5;
    static constexpr int kOffMisc = kOffBars + kNumBars * 8;
    static constexpr int kOffPieces = kOffMisc + 64;
    static constexpr int kSmemBytes = kOffPieces + kMaxPieces * (int)sizeof(Piece) + 1024;  // + alignment slack
    static_assert(NTOK == 16 || NTOK == 32, "token tile is 16 or 32");
    static_assert(kXBoxBytes % 1024 == 0, "x boxes must stay 1024-byte aligned for the 128-byte swizzle");
    static_assert(kOffW % 128 == 0 && kOffEsc % 16 == 0 && kOffHdr % 16 == 0, "copy destinations aligned");
    static_assert(kACol + kASlots * 128 <= kTmemCols && kDCol + 64 <= kACol, "TMEM columns");
    static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM must fit");
    static_assert(Q8 || kESlots == kStages + 1, "an escape slot is reused once the next weight stage is released");
};

struct TcSmBars {
    uint64_t *wfull, *wempty, *efull, *xfull, *xempty, *afull, *aempty, *dfull, *dempty, *hdr, *drain, *epi_in,
        *epi_out, *fin;
};

// ------------------------------------------------------------------ producers
// Weights: the segment headers of the whole range, then per segment its
// packed chunks (one stage) and its escape bytes (one escape slot; only the
// headers decide them, so they need nothing from the other rings).
template <class C>
__device__ void tcsm_producer(const GemmGroup &g, const Piece *pieces, int npieces, uint8_t *smem,
                              const TcSmBars &b, volatile uint32_t *abort_flag, uint64_t deadline) {
    uint8_t *hdr = smem + C::kOffHdr;
    const uint64_t stream_policy = policy_evict_first();  // the weights are read once
    uint32_t hbytes = 0;
    if constexpr (!C::kQ8)
        for (int k = 0; k < npieces; ++k) hbytes += (uint32_t)(pieces[k].s1 - pieces[k].s0) * kSegHdrBytes;
    mbar_arrive_expect_tx(b.hdr, hbytes);  // a Q8 copy has no segment headers
    for (int k = 0, off = 0; !C::kQ8 && k < npieces; ++k) {
        const Piece &pc = pieces[k];
        const GemmParams &p = g.m[pc.member];
        const uint32_t n = (uint32_t)(pc.s1 - pc.s0) * kSegHdrBytes;
        bulk_g2s(hdr + off, p.blob + p.off_seg + (uint64_t)(pc.tile * p.segs + pc.s0) * kSegHdrBytes, n, b.hdr);
        off += (int)n;
    }

    bool hdr_ready = false, failed = false;
    int gw = 0, ge = 0;  // weight stages and escape slots issued (one each per segment)
    int hseg = 0;        // headers of the earlier pieces
    for (int k = 0; !failed && k < npieces; ++k) {
        const Piece &pc = pieces[k];
        const GemmParams &p = g.m[pc.member];
        for (int sg = pc.s0; sg < pc.s1; ++sg) {
            const int chunk = sg * kChunksPerSeg;
            const int nch = min(kChunksPerSeg, p.chunks - chunk);
            const int wslot = gw % C::kStages, eslot = ge % C::kESlots;
            if (gw >= C::kStages && !mbar_wait(b.wempty + wslot, (uint32_t)(gw / C::kStages - 1) & 1u, deadline)) {
                failed = true;
                break;
            }
            mbar_arrive_expect_tx(b.wfull + wslot, (uint32_t)(nch * C::kChunkB));
            bulk_g2s_hint(smem + C::kOffW + wslot * C::kWBytes,
                          p.blob + p.off_w + (uint64_t)(pc.tile * p.chunks + chunk) * C::kChunkB,
                          (uint32_t)(nch * C::kChunkB), b.wfull + wslot, stream_policy);
            ++gw;
            if constexpr (C::kQ8) {
                if (*abort_flag) {
                    failed = true;
                    break;
                }
                continue;  // no headers, no escapes
            }
            if (!hdr_ready) {
                if (!mbar_wait(b.hdr, 0, deadline)) {
                    failed = true;
                    break;
                }
                hdr_ready = true;
            }
            // escape slot gs mod kESlots last held segment gs - kESlots; every
            // decoder finished it before loading segment gs - kESlots + 1,
            // whose weight stage this thread has just seen released (the ring
            // is one stage shorter than the escape slots), so it is free
            const uint4 meta = *reinterpret_cast<const uint4 *>(hdr + (hseg + sg - pc.s0) * kSegHdrBytes + 16);
            const uint32_t base = meta.x;
            const uint32_t total = seg_escape_total(meta);
            if (escapes_staged<C>(total)) {
                const uint32_t src0 = base & ~15u;
                const uint32_t ebytes = ((base + total + 15u) & ~15u) - src0;
                mbar_arrive_expect_tx(b.efull + eslot, ebytes);
                bulk_g2s(smem + C::kOffEsc + eslot * C::kEscCap, p.blob + p.off_esc + src0, ebytes, b.efull + eslot);
            } else {
                mbar_arrive(b.efull + eslot);
            }
            ++ge;
            if (*abort_flag) {
                failed = true;
                break;
            }
        }
        hseg += pc.s1 - pc.s0;
    }
    if (failed && !*abort_flag) raise_timeout(group_status(g), abort_flag);
    if (failed) {
        // let every copy still in flight land before the CTA can exit
        const uint64_t drain_deadline = globaltimer_ns() + 1000000000ull;
        for (int st = max(0, gw - C::kStages); st < gw; ++st)
            mbar_wait(b.wfull + st % C::kStages, (uint32_t)(st / C::kStages) & 1u, drain_deadline);
        mbar_wait(b.hdr, 0, drain_deadline);
        for (int se = max(0, ge - C::kESlots); se < ge; ++se)
            mbar_wait(b.efull + se % C::kESlots, (uint32_t)(se / C::kESlots) & 1u, drain_deadline);
    }
}

// x: per segment the 256-column tile of the token rows (four 64-column boxes,
// 128-byte swizzle, rows past M and columns past K zero-filled by the tensor
// copy); a slot is free again once the MMAs that read it have completed.
template <class C>
__device__ void tcsm_x_loader(const GemmGroup &g, const Piece *pieces, int npieces, const CUtensorMap *tmap,
                              uint8_t *smem, const TcSmBars &b, volatile uint32_t *abort_flag, uint64_t deadline) {
    prefetch_tmap(tmap);
    bool failed = false;
    int gs = 0;
    for (int k = 0; !failed && k < npieces; ++k) {
        const Piece &pc = pieces[k];
        for (int sg = pc.s0; sg < pc.s1; ++sg) {
            const int xslot = gs % C::kXSlots;
            if (gs >= C::kXSlots && !mbar_wait(b.xempty + xslot, (uint32_t)(gs / C::kXSlots - 1) & 1u, deadline)) {
                failed = true;
                break;
            }
            mbar_arrive_expect_tx(b.xfull + xslot, (uint32_t)C::kXBytes);
            uint8_t *xs = smem + C::kOffX + xslot * C::kXBytes;
#pragma unroll
            for (int bx = 0; bx < 4; ++bx)
                tma_load_2d(xs + bx * C::kXBoxBytes, tmap, sg * kSegK + bx * 64, 0, b.xfull + xslot);
            ++gs;
            if (*abort_flag) {
                failed = true;
                break;
            }
        }
    }
    if (*abort_flag || failed) {
        if (!*abort_flag) raise_timeout(group_status(g), abort_flag);
        const uint64_t drain_deadline = globaltimer_ns() + 1000000000ull;
        for (int sx = max(0, gs - C::kXSlots); sx < gs; ++sx)
            mbar_wait(b.xfull + sx % C::kXSlots, (uint32_t)(sx / C::kXSlots) & 1u, drain_deadline);
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
            const int xslot = gs % C::kXSlots, aslot = gs % C::kASlots;
            if (!mbar_wait(b.xfull + xslot, (uint32_t)(gs / C::kXSlots) & 1u, deadline) ||
                !mbar_wait(b.afull + aslot, (uint32_t)(gs / C::kASlots) & 1u, deadline)) {
                failed = true;
                break;
            }
            tc_fence_after();
            // one descriptor per segment: a k-block's B starts kb / 4 boxes and
            // 32 (kb mod 4) bytes further on, i.e. a constant added to the
            // descriptor's start-address field (16-byte units, no carry: shared
            // addresses stay below 2^18)
            const uint64_t bdesc0 = smem_desc(smem_u32(smem + C::kOffX + xslot * C::kXBytes), 16u, 1024u, 2u);
            const uint32_t a_taddr = tmem_base + (uint32_t)(C::kACol + 128 * aslot);
            const uint32_t acc0 = sg > pc.s0 ? 1u : 0u;
            if (nch == kChunksPerSeg) {
                // the common full segment: sixteen MMAs with constant offsets,
                // so the issuing thread spends its issue slots on MMAs
#pragma unroll
                for (int kb = 0; kb < 2 * kChunksPerSeg; ++kb)
                    mma_tmem_a(d_taddr, a_taddr + (uint32_t)(8 * kb),
                               bdesc0 + (uint64_t)((kb >> 2) * (C::kXBoxBytes >> 4) + (kb & 3) * 2), idesc,
                               kb > 0 ? 1u : acc0);
            } else {
                for (int kb = 0; kb < 2 * nch; ++kb)
                    mma_tmem_a(d_taddr, a_taddr + (uint32_t)(8 * kb),
                               bdesc0 + (uint64_t)((kb >> 2) * (C::kXBoxBytes >> 4) + (kb & 3) * 2), idesc,
                               kb > 0 ? 1u : acc0);
            }
            mma_commit(b.aempty + aslot);
            mma_commit(b.xempty + xslot);
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

// ------------------------------------------------------------------ finish
// A tile whose last arrival this CTA made at the end of its range, added up
// from memory: every output adds the tile's slots in slot order (reproducible
// run to run) and is rounded to BF16.  The decode and epilogue warps share
// the outputs (reducer id rid of kFinishThreads), four per thread per batch
// with up to four slots each in flight: at the end of the kernel every load
// waits behind the weight stream of the SMs still working.
template <class C>
__device__ void tcsm_finish(const GemmParams &p, const Piece &pc, int rid) {
    constexpr int kN = C::kFinishThreads;
    const int total = p.M * kTileRows;
    const int64_t stride = (int64_t)p.M * p.Npad;
    const float *base = p.partials + pc.tile * kTileRows;
    // a warp's 32 outputs share one token (kN and 128 are multiples of 32)
    for (int o0 = rid; o0 < total; o0 += 4 * kN) {
        float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int sp0 = 0; sp0 < pc.count; sp0 += 4) {
            float v[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int bb = 0; bb < 4; ++bb) {
                    const int o = o0 + bb * kN;
                    v[u][bb] = (sp0 + u < pc.count && o < total)
                                   ? __ldcg(base + (int64_t)(sp0 + u) * stride + (int64_t)(o / kTileRows) * p.Npad +
                                            o % kTileRows)
                                   : 0.0f;
                }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int bb = 0; bb < 4; ++bb)
                    if (sp0 + u < pc.count) s[bb] += v[u][bb];
        }
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
            const int o = o0 + bb * kN;
            if (o >= total) break;  // the same for the whole warp
            const int t = o / kTileRows;
            const int64_t n = pc.tile * kTileRows + o % kTileRows;
            if constexpr (C::kQ8) s[bb] *= p.scales[n];  // the Q8 copy's row scale (pad rows: 0)
            if (p.y != nullptr && n < p.N) p.y[(int64_t)t * p.N + n] = bf16_bits_rn(s[bb]);
            if (p.amax != nullptr) argmax_warp(p.amax + t, n < p.N ? argmax_key(s[bb], (uint32_t)n) : 0ull);
        }
    }
}

// The range's tiles that this CTA completed as their last arrival: bit 0 the
// first piece's tile, bit 1 the last piece's.
template <class C>
__device__ __noinline__ void tcsm_finish_all(const GemmGroup &g, const Piece *pieces, int npieces, int mask,
                                             int rid) {
    if (mask & 1) tcsm_finish<C>(g.m[pieces[0].member], pieces[0], rid);
    if (mask & 2) tcsm_finish<C>(g.m[pieces[npieces - 1].member], pieces[npieces - 1], rid);
}

// The decode warps after their last segment: the epilogue says, once per
// launch, whether tiles of the range must be added up from memory, and then
// every decode warp helps.  Kept out of line: what the decode loop keeps live
// for code after it costs the loop registers, and it measured slower inline.
template <class C>
__device__ __noinline__ void tcsm_decoder_finish(const GemmGroup &g, const Piece *pieces, int npieces, uint64_t *fin,
                                                 volatile int *fin_mask, volatile uint32_t *abort_flag,
                                                 uint64_t deadline) {
    if (!warp_wait(fin, 0, deadline)) {
        if ((threadIdx.x & 31) == 0) raise_timeout(group_status(g), abort_flag);
        return;
    }
    tcsm_finish_all<C>(g, pieces, npieces, *fin_mask, (int)threadIdx.x);
}

// ------------------------------------------------------------------ decoders
// Decode one chunk of this thread's row and store its 32 weights as 16 TMEM
// columns of BF16 pairs (column c: weights 2c, 2c + 1) at taddr.
__device__ __forceinline__ void decode_chunk_to_tmem(const Table &T, const uint4 &s0, const uint4 &s1,
                                                     const uint4 &cd, bool has_escapes, const uint8_t *&run,
                                                     uint32_t taddr) {
    uint32_t v[16];
    decode_chunk_patched(T, s0, s1, cd, has_escapes, run, v);
    tmem_st16(taddr, v);
}

template <class C>
__device__ void tcsm_decode(const GemmGroup &g, const Piece *pieces, int npieces, uint8_t *smem, const TcSmBars &b,
                            volatile uint32_t *abort_flag, volatile int *fin_mask, uint32_t tmem_base,
                            uint64_t deadline) {
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
    for (int k = 0; ok && k < npieces; ++k) {
        const Piece &pc = pieces[k];
        const GemmParams &p = g.m[pc.member];
        for (int sg = pc.s0; sg < pc.s1; ++sg, ++gs) {
            const int nch = min(kChunksPerSeg, p.chunks - sg * kChunksPerSeg);
            const uint8_t *hp = hdr + (hseg + sg - pc.s0) * kSegHdrBytes;
            const Table T = make_table(*reinterpret_cast<const uint4 *>(hp));
            const uint4 meta = *reinterpret_cast<const uint4 *>(hp + 16);
            const uint32_t mask_q = (meta.w >> (8 * q)) & 0xFFu;
            const int eslot = gs % C::kESlots, wslot = gs % C::kStages;
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
            if (esc_a | esc_b) {
                const uint32_t pos = quarter_chunk_escape_pos(meta, q, j, mask_q, nch, acd, bcd, esc_a, esc_b, sw);
                if (!(ok = warp_wait(b.efull + eslot, (uint32_t)(gs / C::kESlots) & 1u, deadline))) break;
                if (escapes_staged<C>(seg_escape_total(meta)))
                    run = smem + C::kOffEsc + eslot * C::kEscCap + (meta.x & 15u) + pos;
                else
                    run = p.blob + p.off_esc + meta.x + pos;
            }
            warp_arrive(b.wempty + wslot);  // this warp is done with the stage's bytes

            const int aslot = gs % C::kASlots;
            if (gs >= C::kASlots &&
                !(ok = warp_wait(b.aempty + aslot, (uint32_t)(gs / C::kASlots - 1) & 1u, deadline)))
                break;
            tc_fence_after();
            // a chunk goes to TMEM as 16 columns of BF16 pairs, its 32 weights
            // in column order
            const uint32_t ta = a_lane + (uint32_t)(128 * aslot);
            // (each chunk is stored as soon as it is decoded: decoding both
            // chunks first and storing them together measured slower)
            if (va) decode_chunk_to_tmem(T, a0, a1, acd, esc_a != 0u, run, ta);
            if (vb) decode_chunk_to_tmem(T, b0, b1, bcd, esc_b != 0u, run, ta + 16u);
            // hand the slot to the MMA warp once the stores have landed (doing
            // this one segment later, to overlap the store latency with the
            // next loads, measured slower: the MMAs then start a segment later
            // and the decoders wait for the slot three segments on)
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(b.afull + aslot);
            if (*abort_flag) {
                ok = false;
                break;
            }
        }
        hseg += pc.s1 - pc.s0;
    }
    if (!ok) {
        tmem_wait_st();  // no store of this warp may still be in flight when TMEM is freed
        if (lane == 0) raise_timeout(group_status(g), abort_flag);
        return;
    }
    tcsm_decoder_finish<C>(g, pieces, npieces, b.fin, fin_mask, abort_flag, deadline);
}

// The Q8 copy: chunk 2j and 2j + 1 of this thread's row as 16 int8 per slab,
// turned into BF16 exactly (|q| <= 127) and stored like the W12 weights.
template <class C>
__device__ void tcsm_decode_q8(const GemmGroup &g, const Piece *pieces, int npieces, uint8_t *smem,
                               const TcSmBars &b, volatile uint32_t *abort_flag, volatile int *fin_mask,
                               uint32_t tmem_base, uint64_t deadline) {
    const int warp = threadIdx.x >> 5;
    const int q = warp & 3;
    const int j = warp >> 2;
    const int lane = threadIdx.x & 31;
    const int r = 32 * q + lane;
    const uint32_t s_row = smem_u32(smem + C::kOffW) + (uint32_t)(16 * r);
    const uint32_t a_lane = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(C::kACol + 32 * j);
    bool ok = true;
    int gs = 0;
    for (int k = 0; ok && k < npieces; ++k) {
        const Piece &pc = pieces[k];
        const GemmParams &p = g.m[pc.member];
        for (int sg = pc.s0; sg < pc.s1; ++sg, ++gs) {
            const int nch = min(kChunksPerSeg, p.chunks - sg * kChunksPerSeg);
            const int wslot = gs % C::kStages, aslot = gs % C::kASlots;
            if (!(ok = warp_wait(b.wfull + wslot, (uint32_t)(gs / C::kStages) & 1u, deadline))) break;
            const int ca = 2 * j;
            const bool va = ca < nch, vb = ca + 1 < nch;
            const uint32_t sa = s_row + (uint32_t)(wslot * C::kWBytes + ca * C::kChunkB);
            uint4 a0{}, a1{}, b0{}, b1{};
            if (va) {
                a0 = lds128(sa);
                a1 = lds128(sa + kSlabBytes);
            }
            if (vb) {
                b0 = lds128(sa + C::kChunkB);
                b1 = lds128(sa + C::kChunkB + kSlabBytes);
            }
            warp_arrive(b.wempty + wslot);
            if (gs >= C::kASlots &&
                !(ok = warp_wait(b.aempty + aslot, (uint32_t)(gs / C::kASlots - 1) & 1u, deadline)))
                break;
            tc_fence_after();
            const uint32_t ta = a_lane + (uint32_t)(128 * aslot);
            if (va) {
                uint32_t lo[8], hi[8], v[16];
                q8_half(a0, lo);
                q8_half(a1, hi);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    v[i] = lo[i];
                    v[8 + i] = hi[i];
                }
                tmem_st16(ta, v);
            }
            if (vb) {
                uint32_t lo[8], hi[8], v[16];
                q8_half(b0, lo);
                q8_half(b1, hi);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    v[i] = lo[i];
                    v[8 + i] = hi[i];
                }
                tmem_st16(ta + 16u, v);
            }
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(b.afull + aslot);
            if (*abort_flag) {
                ok = false;
                break;
            }
        }
    }
    if (!ok) {
        tmem_wait_st();
        if (lane == 0) raise_timeout(group_status(g), abort_flag);
        return;
    }
    tcsm_decoder_finish<C>(g, pieces, npieces, b.fin, fin_mask, abort_flag, deadline);
}

// ------------------------------------------------------------------ epilogue
// The four epilogue warps meet on an mbarrier pair (in: four arrivals, out:
// the leader's) at most twice per launch; `use` counts the meetings so the
// phases line up.
struct EpiSync {
    uint64_t *in, *out;
    int use;
};

// Add the partial-sum slots of a tile in slot order (run-to-run reproducible)
// and store the BF16 result: row r of the tile, tokens 0..M-1.  The slot
// `own` (or none, when own < 0) comes from `acc` instead of memory.  Eight
// tokens' loads of a slot are in flight together.
template <int NT, bool Q8>
__device__ __forceinline__ void tcsm_reduce_row(const GemmParams &p, const Piece &pc, int r, int own,
                                                float (&acc)[NT]) {
    constexpr int kB = 8;  // tokens per batch (register budget of the epilogue)
    const int64_t n = pc.tile * kTileRows + r;
    const float sc = Q8 ? p.scales[n] : 1.0f;  // the Q8 copy's row scale (pad rows: 0)
    const float *src = p.partials + (n < p.N ? n : pc.tile * kTileRows);
    if (own == 0) {
        // this CTA holds slot 0 (the usual case: it computed the tile's first
        // segments at the end of its range): add the other slots onto the
        // registers in slot order, sixteen tokens' loads in flight at a time
        for (int sp = 1; sp < pc.count; ++sp) {
#pragma unroll
            for (int t0 = 0; t0 < NT; t0 += 16) {
                if (t0 >= p.M) break;
                float v[16];
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    v[u] = t0 + u < p.M ? __ldcg(src + ((int64_t)sp * p.M + t0 + u) * p.Npad) : 0.0f;
#pragma unroll
                for (int u = 0; u < 16; ++u) acc[t0 + u] += v[u];
            }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (t >= p.M) break;
            const float v = Q8 ? acc[t] * sc : acc[t];
            if (p.y != nullptr && n < p.N) p.y[(int64_t)t * p.N + n] = bf16_bits_rn(v);
            if (p.amax != nullptr) argmax_warp(p.amax + t, n < p.N ? argmax_key(v, (uint32_t)n) : 0ull);
        }
        return;
    }
#pragma unroll
    for (int t0 = 0; t0 < NT; t0 += kB) {
        if (t0 >= p.M) break;
        float s[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) s[u] = 0.0f;
        for (int sp = 0; sp < pc.count; ++sp) {
            float v[kB];
            if (sp == own) {
#pragma unroll
                for (int u = 0; u < kB; ++u) v[u] = acc[t0 + u];
            } else {
#pragma unroll
                for (int u = 0; u < kB; ++u)
                    v[u] = t0 + u < p.M ? __ldcg(src + ((int64_t)sp * p.M + t0 + u) * p.Npad) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < kB; ++u) s[u] += v[u];
        }
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const int t = t0 + u;
            if (t >= p.M) break;
            if (Q8) s[u] *= sc;
            if (p.y != nullptr && n < p.N) p.y[(int64_t)t * p.N + n] = bf16_bits_rn(s[u]);
            if (p.amax != nullptr) argmax_warp(p.amax + t, n < p.N ? argmax_key(s[u], (uint32_t)n) : 0ull);
        }
    }
}

// One warp per TMEM lane quarter.  For each piece: wait for its accumulator,
// read this quarter's 32 rows x NTOK tokens, release the accumulator, then
//   - a whole tile: store y;
//   - a shared tile that is not the range's last piece (it was computed
//     early, while the CTAs sharing it are still busy): store the partial-sum
//     slot and arrive on the tile's counter at once (a release fence, then one
//     atomic add);
//   - the range's last piece, shared: the other CTAs normally arrived long
//     ago, so first look (acquire load of the counter): if they all have,
//     add their slots to this accumulator, still in registers, and store y,
//     with no partial store, fence or atomic on the kernel's tail; otherwise
//     store the slot and arrive as above.
// The last arrival of a tile resets its counter for the next call; a tile it
// must add up from memory is left for the end of the range, where the decode
// warps (done by then) share the loads.
template <class C>
__device__ void tcsm_epilogue(const GemmGroup &g, const Piece *pieces, int npieces, const TcSmBars &b,
                              volatile uint32_t *abort_flag, volatile uint32_t *flag, volatile int *fin_mask,
                              uint32_t tmem_base, uint64_t deadline) {
    constexpr int NT = C::kNtok;
    const int warp = threadIdx.x >> 5;
    const int q = warp & 3;
    const int lane = threadIdx.x & 31;
    const int r = 32 * q + lane;
    const bool leader = warp == C::kEpiWarp0 && lane == 0;
    const uint32_t d_lane = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)C::kDCol;
    EpiSync sy{b.epi_in, b.epi_out, 0};
    // all four warps meet; the leader runs `lead` in between and writes its
    // result to *flag, which every warp reads after the meeting
    auto meet = [&](auto lead) -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(sy.in);
        if (leader) {
            if (mbar_wait(sy.in, (uint32_t)sy.use & 1u, deadline)) {
                *flag = lead() ? 1u : 0u;
                mbar_arrive(sy.out);
            } else {
                raise_timeout(group_status(g), abort_flag);
            }
        }
        const bool ok = warp_wait(sy.out, (uint32_t)sy.use & 1u, deadline);
        ++sy.use;
        return ok;
    };
    for (int k = 0; k < npieces; ++k) {
        const Piece &pc = pieces[k];
        const GemmParams &p = g.m[pc.member];
        const int dbuf = k & 1;
        bool ok = warp_wait(b.dfull + dbuf, (uint32_t)(k >> 1) & 1u, deadline);
        if (!ok) {
            if (lane == 0) raise_timeout(group_status(g), abort_flag);
            return;
        }
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
            const float sc = C::kQ8 ? p.scales[n] : 1.0f;  // the Q8 copy's row scale (pad rows: 0)
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                if (C::kQ8) acc[t] *= sc;
                if (t < p.M) {
                    if (p.y != nullptr && n < p.N) p.y[(int64_t)t * p.N + n] = bf16_bits_rn(acc[t]);
                    if (p.amax != nullptr) argmax_warp(p.amax + t, n < p.N ? argmax_key(acc[t], (uint32_t)n) : 0ull);
                }
            }
            continue;
        }
        uint32_t *counter = p.counters + pc.tile;
        if (k == npieces - 1) {
            // everyone else in already?  Then add up straight from registers
            ok = meet([&] { return load_acquire_gpu(counter) == (uint32_t)(pc.count - 1); });
            if (!ok) return;
            if (*flag) {
                tcsm_reduce_row<NT, C::kQ8>(p, pc, r, pc.idx, acc);
                if (leader) *counter = 0u;  // every CTA of the tile has arrived
                continue;
            }
        }
        // store this piece's slot, then arrive: the mbarrier meeting orders the
        // four warps' stores before the leader's release fence
#pragma unroll
        for (int t = 0; t < NT; ++t)
            if (t < p.M) __stcg(p.partials + ((int64_t)pc.idx * p.M + t) * p.Npad + n, acc[t]);
        ok = meet([&] {
            fence_acq_rel_gpu();
            const bool last = arrive_relaxed(counter) == (uint32_t)(pc.count - 1);
            if (last) fence_acq_rel_gpu();
            return last;
        });
        if (!ok) return;
        // last arrival: the tile is added up from memory at the end of the
        // range, by the decode and epilogue warps together (even a first
        // piece's tile: its sharers arrive at the ends of their ranges, so
        // this is near the end anyway)
        if (*flag && leader) {
            *counter = 0u;
            *fin_mask |= k == 0 ? 1 : 2;
        }
    }
    // tell the decode warps whether there is a finish to share (exactly once
    // per launch, also when there is nothing to do)
    __syncwarp();
    if (leader) mbar_arrive(b.fin);
    if (!warp_wait(b.fin, 0, deadline)) return;
    tcsm_finish_all<C>(g, pieces, npieces, *fin_mask, (int)threadIdx.x - (C::kEpiWarp0 - C::kDecWarps) * 32);
}

// ------------------------------------------------------------------ kernel
template <int NTOK, bool Q8 = false>
__global__ void __launch_bounds__(TcSmCfg<NTOK, Q8>::kThreads, 1)
    w12_gemm_tc_sm_kernel(const __grid_constant__ GemmGroup grp, const __grid_constant__ CUtensorMap tmap_x) {
    using C = TcSmCfg<NTOK, Q8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBars);
    TcSmBars b;
    b.wfull = bars;
    b.wempty = b.wfull + C::kStages;
    b.efull = b.wempty + C::kStages;
    b.xfull = b.efull + C::kESlots;
    b.xempty = b.xfull + C::kXSlots;
    b.afull = b.xempty + C::kXSlots;
    b.aempty = b.afull + C::kASlots;
    b.dfull = b.aempty + C::kASlots;
    b.dempty = b.dfull + 2;
    b.hdr = b.dempty + 2;
    b.drain = b.hdr + 1;
    b.epi_in = b.drain + 1;
    b.epi_out = b.epi_in + 1;
    b.fin = b.epi_out + 1;
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    uint32_t *tmem_slot = misc;
    volatile uint32_t *abort_flag = misc + 1;
    volatile uint32_t *npieces = misc + 2;
    volatile uint32_t *last_flags = misc + 4;  // the epilogue leader's word to the other epilogue warps
    volatile int *fin_mask = reinterpret_cast<volatile int *>(misc + 5);  // tiles to add up at the end
    Piece *pieces = reinterpret_cast<Piece *>(smem + C::kOffPieces);

    const int warp = threadIdx.x >> 5;
    const uint64_t deadline = globaltimer_ns() + grp.m[0].timeout_ns;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(b.wfull + i, 1);
            mbar_init(b.wempty + i, C::kDecWarps);
        }
        for (int i = 0; i < C::kESlots; ++i) mbar_init(b.efull + i, 1);
        for (int i = 0; i < C::kXSlots; ++i) {
            mbar_init(b.xfull + i, 1);
            mbar_init(b.xempty + i, 1);  // the MMAs that read the slot have completed
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
        mbar_init(b.fin, 1);
        *abort_flag = 0u;
        last_flags[0] = 0u;
        *fin_mask = 0;
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
    if (warp == C::kProdWarp && (threadIdx.x & 31) == 0) prefetch_pieces<C::kChunkB, !Q8>(grp, pieces, np);
    pdl_wait();

    if (warp == C::kProdWarp) {
        if ((threadIdx.x & 31) == 0) tcsm_producer<C>(grp, pieces, np, smem, b, abort_flag, deadline);
    } else if (warp == C::kXWarp) {
        if ((threadIdx.x & 31) == 0) tcsm_x_loader<C>(grp, pieces, np, &tmap_x, smem, b, abort_flag, deadline);
    } else if (warp == C::kMmaWarp) {
        if ((threadIdx.x & 31) == 0) tcsm_mma<C>(grp, pieces, np, smem, b, abort_flag, tmem_base, deadline);
        __syncwarp();
    } else if (warp >= C::kEpiWarp0 && warp < C::kEpiWarp0 + C::kEpiWarps) {
        tcsm_epilogue<C>(grp, pieces, np, b, abort_flag, last_flags, fin_mask, tmem_base, deadline);
    } else {
        if constexpr (Q8)
            tcsm_decode_q8<C>(grp, pieces, np, smem, b, abort_flag, fin_mask, tmem_base, deadline);
        else
            tcsm_decode<C>(grp, pieces, np, smem, b, abort_flag, fin_mask, tmem_base, deadline);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::kMmaWarp) tmem_dealloc(tmem_base, C::kTmemCols);
}

}  // namespace dev
}  // namespace w12
