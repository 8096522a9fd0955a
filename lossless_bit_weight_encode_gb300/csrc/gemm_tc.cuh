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
// Warp roles (320 threads):
//   warps 0-7  decode: warp w handles rows 32q..32q+31 (q = w mod 4, the TMEM
//              lanes of quarter q) and columns 16h..16h+15 of every chunk
//              (h = w / 4); per weight stage (2 chunks) a thread reads its
//              row's S bytes and codes from SMEM, decodes 2 x 16 weights,
//              patches escapes and stores 2 x 8 columns of BF16 pairs into a
//              TMEM A slot (or SMEM A slot); one handshake with the MMA warp
//              per stage; afterwards the warp runs the epilogue for half of
//              the token columns;
//   warp 8     producer: one lane issues cp.async.bulk for the segment
//              headers and for every weight stage (2 packed chunks, 12 KB), and
//              per segment cp.async.bulk.tensor for the segment's 256-column x
//              tile (four 64-column boxes, 128-byte swizzle) plus
//              cp.async.bulk for the segment's escape bytes;
//   warp 9     allocates TMEM; one lane issues tcgen05.mma (2 per chunk) and
//              tcgen05.commit.
// Rings: weight stages are released by the decode warps as soon as they have
// read them (no MMA latency in that loop); the per-segment x tile and escape
// bytes are released when the segment's MMAs have completed and its decoders
// are done.  Waits are made by one lane per warp; __syncwarp orders the rest.
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
    uint16_t *y;              // [M][N] BF16 (may be null when amax is set)
    unsigned long long *amax; // [M] argmax keys (null: plain GEMM)
    const float *scales;      // [Npad] per-row scales of a Q8 copy (null: W12)
    uint32_t *status;         // device status word
    uint64_t timeout_ns;
};

// Up to kMaxGroup matrices that share x (and so K) in one launch: group tile
// y (all members' tiles in order) belongs to matrix i when tile0[i] <= y <
// tile0[i + 1]; each matrix keeps its own blob, output, partials and counters.
//
// Two ways to share the work among CTAs.  Fixed split-K (units == 0): grid
// (splits, tiles); CTA (x, y) takes segments [x segs / splits, (x + 1) segs /
// splits) of group tile y.  Stream-K (units > 0): the group's tiles, each cut
// into its segs segments, form one sequence of units = tiles x segs; CTA c of
// the 1-D grid of ctas takes units [c units / ctas, (c + 1) units / ctas), a
// range that may end one tile and start the next, so that a single wave of
// CTAs gets equal work however the tile count divides the SM count.  The
// planner keeps units x ctas below 2^31, so this arithmetic is 32-bit.
constexpr int kMaxGroup = 4;
struct GemmGroup {
    GemmParams m[kMaxGroup];
    int64_t tile0[kMaxGroup + 1];
    int32_t units;  // stream-K units (0: fixed split-K)
    int32_t ctas;   // stream-K grid size
    int32_t n;
};

// Every member reports to the same device status word.
__device__ __forceinline__ uint32_t *group_status(const GemmGroup &g) { return g.m[0].status; }

// The member holding group tile gt and the tile's index within it.
__device__ __forceinline__ int member_of(const GemmGroup &g, int64_t gt, int64_t *tile) {
    int i = 0;
#pragma unroll
    for (int j = 1; j < kMaxGroup; ++j)
        if (j < g.n && gt >= g.tile0[j]) i = j;
    *tile = gt - g.tile0[i];
    return i;
}

// The matrix of this CTA's grid row and the row's tile within it (fixed split-K).
__device__ __forceinline__ int group_member(const GemmGroup &g, int64_t *tile) {
    return member_of(g, (int64_t)blockIdx.y, tile);
}

// One CTA's share of one tile: segments [s0, s1), partial-sum slot idx of the
// tile's count shares (count == 1: the CTA owns the whole tile).
struct Piece {
    int member;
    int64_t tile;  // within the member
    int s0, s1;
    int idx, count;
};

// The units of this CTA still to hand out as pieces.
struct CtaWork {
    uint32_t u, u1;
};

__device__ __forceinline__ CtaWork cta_work(const GemmGroup &g) {
    if (g.units == 0) return CtaWork{0u, 1u};
    const uint32_t c = blockIdx.x, units = (uint32_t)g.units, ctas = (uint32_t)g.ctas;
    return CtaWork{c * units / ctas, (c + 1u) * units / ctas};
}

// The stream-K CTA whose range holds unit u: the largest c with
// floor(c units / ctas) <= u.
__device__ __forceinline__ uint32_t unit_owner(const GemmGroup &g, uint32_t u) {
    return ((u + 1u) * (uint32_t)g.ctas - 1u) / (uint32_t)g.units;
}

// The next piece of this CTA's work, in order; false when none is left.
__device__ __forceinline__ bool next_piece(const GemmGroup &g, CtaWork &w, Piece &pc) {
    if (w.u >= w.u1) return false;
    if (g.units == 0) {
        pc.member = group_member(g, &pc.tile);
        const GemmParams &p = g.m[pc.member];
        pc.idx = (int)blockIdx.x;
        pc.count = p.splits;
        pc.s0 = (int)((int64_t)pc.idx * p.segs / p.splits);
        pc.s1 = (int)((int64_t)(pc.idx + 1) * p.segs / p.splits);
        w.u = w.u1;
        return true;
    }
    const uint32_t segs = (uint32_t)g.m[0].segs;
    const uint32_t gt = w.u / segs, first_unit = gt * segs;
    pc.s0 = (int)(w.u - first_unit);
    pc.s1 = (int)min(segs, w.u1 - first_unit);
    if (pc.s0 == 0 && first_unit + segs <= w.u1) {
        pc.idx = 0;  // the whole tile lies in this range
        pc.count = 1;
    } else {
        const uint32_t first = unit_owner(g, first_unit);
        pc.idx = (int)(blockIdx.x - first);
        pc.count = (int)(unit_owner(g, first_unit + segs - 1u) - first + 1u);
    }
    pc.member = member_of(g, (int64_t)gt, &pc.tile);
    w.u = first_unit + (uint32_t)pc.s1;
    return true;
}

template <int NTOK, int STAGES, bool A_SMEM, bool Q8 = false>
struct GemmCfg {
    static constexpr bool kQ8 = Q8;                             // weights: Q8 copy instead of W12
    static constexpr int kChunkB = Q8 ? q8::kChunkBytes : kChunkBytes;
    static constexpr int kThreads = 320;
    static constexpr int kDecWarps = 8;
    static constexpr int kStages = STAGES;
    static constexpr bool kASmem = A_SMEM;
    static constexpr int kNtok = NTOK;
    static constexpr int kWBytes = 2 * kChunkB;                 // weight stage: 2 chunks
    static constexpr int kXBoxBytes = NTOK * 128;               // one 64-column x box
    static constexpr int kXBytes = 4 * kXBoxBytes;              // x tile of one segment
    static constexpr int kSegSlots = 2;                         // x + escapes per segment
    // TMEM A slots, one weight stage (2 chunks) each: four for the 32-token
    // tile (two CTAs per SM, 256 TMEM columns each; measured 1.5 % faster than
    // three, and six were slower), three for the 16-token tile (three CTAs per
    // SM, 128 columns each)
    static constexpr int kASlots = NTOK == 32 ? 4 : 3;
    static constexpr int kASlotBytes = 2 * kTileRows * kChunkK * 2;  // 16 KB (SMEM A variant)
    static constexpr int kAChunkBytes = kTileRows * kChunkK * 2;     // 8 KB per chunk
    static constexpr int kEscCap = Q8 ? 0 : 2048;
    static constexpr int kMaxSegs = 96;   // segments per CTA (K range <= 24576)
    static constexpr int kTmemCols = NTOK == 32 ? 256 : 128;
    static constexpr int kDCol = 0;
    static constexpr int kACol = 32;
    static constexpr int kOffX = 0;                                         // 1024-aligned
    static constexpr int kOffW = kOffX + kSegSlots * kXBytes;
    static constexpr int kOffA = kOffW + STAGES * kWBytes;
    static constexpr int kOffEsc = kOffA + (A_SMEM ? kASlots * kASlotBytes : 0);
    static constexpr int kOffHdr = kOffEsc + kSegSlots * kEscCap;
    static constexpr int kOffBars = kOffHdr + kMaxSegs * kSegHdrBytes;
    // wfull[S], wempty[S], sfull[2], sempty[2], afull[kASlots], aempty[kASlots],
    // hdr, accum, drain, epi_in, epi_out
    static constexpr int kNumBars = 2 * STAGES + 2 * kSegSlots + 2 * kASlots + 5;
    static constexpr int kOffMisc = kOffBars + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 64 + 1024;  // + slack to align the base to 1024
    static_assert(kXBoxBytes % 1024 == 0, "x boxes must stay 1024-byte aligned for the 128-byte swizzle");
    static_assert(NTOK == 16 || NTOK == 32, "token tile is 16 or 32");
};

struct Bars {
    uint64_t *wfull, *wempty, *sfull, *sempty, *afull, *aempty, *hdr, *accum, *drain, *epi_in, *epi_out;
};

// Whole-warp wait.  Usually the phase has already completed and one try_wait
// by every lane settles it (no branch, no shuffle); otherwise one lane waits
// (bounded), the result is broadcast and __syncwarp orders the other lanes
// after the completed phase.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t deadline) {
    if (__all_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity))) return true;
    uint32_t ok = 0;
    if ((threadIdx.x & 31u) == 0) ok = mbar_wait(bar, parity, deadline) ? 1u : 0u;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    __syncwarp();
    return ok != 0;
}

__device__ __forceinline__ void raise_timeout(uint32_t *status, volatile uint32_t *abort_flag) {
    *abort_flag = 1u;
    atomicOr(status, kStatusTimeout);
}

__device__ __forceinline__ uint16_t bf16_bits_rn(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ uint32_t seg_escape_total(const uint4 &meta) {
    return (meta.y & 0xFFFFu) + (meta.y >> 16) + (meta.z & 0xFFFFu) + (meta.z >> 16);
}

template <class C>
__device__ __forceinline__ bool escapes_staged(uint32_t total) {
    return total > 0 && total + 30u <= (uint32_t)C::kEscCap;
}


// Before waiting for the previous kernel in the stream: pull this CTA's first
// weight bytes (its segment headers and up to kPrefetchBytes of packed chunks)
// into L2.  Only L2 is warmed here; every load that lands in shared memory is
// issued after griddepcontrol.wait, so a blob written by that previous kernel
// is still read correctly.
constexpr uint32_t kPrefetchBytes = 96 * 1024;
template <int kChunkB, bool kHeaders>
__device__ __forceinline__ void prefetch_cta_weights(const GemmParams &p, int64_t tile, int s0, int c0, int c1,
                                                     uint32_t &budget) {
    if (kHeaders) {
        const int nsegs_cta = (c1 - c0 + kChunksPerSeg - 1) / kChunksPerSeg;
        prefetch_l2(p.blob + p.off_seg + (uint64_t)(tile * p.segs + s0) * kSegHdrBytes,
                    (uint32_t)nsegs_cta * kSegHdrBytes);
    }
    const uint8_t *w = p.blob + p.off_w + (uint64_t)(tile * p.chunks + c0) * kChunkB;
    uint32_t left = (uint32_t)(c1 - c0) * kChunkB;
    if (left > budget) left = budget;
    budget -= left;
    for (uint32_t off = 0; off < left; off += 4 * kChunkB) {
        const uint32_t n = left - off < 4u * kChunkB ? left - off : 4u * kChunkB;
        prefetch_l2(w + off, n);
    }
}

// The same for each of a CTA's pieces in order until kPrefetchBytes are asked for.
template <int kChunkB, bool kHeaders>
__device__ __forceinline__ void prefetch_pieces(const GemmGroup &g, const Piece *pieces, int npieces) {
    uint32_t budget = kPrefetchBytes;
    for (int k = 0; k < npieces && budget > 0; ++k) {
        const Piece &pc = pieces[k];
        const GemmParams &p = g.m[pc.member];
        prefetch_cta_weights<kChunkB, kHeaders>(p, pc.tile, pc.s0, pc.s0 * kChunksPerSeg,
                                                min(pc.s1 * kChunksPerSeg, p.chunks), budget);
    }
}

// ------------------------------------------------------------------ producer
template <class C>
__device__ void gemm_producer(const GemmParams &p, const CUtensorMap *tmap, uint8_t *smem, const Bars &b,
                              volatile uint32_t *abort_flag, int64_t tile, int s0, int c0, int c1,
                              uint64_t deadline) {
    const int nchunks = c1 - c0;
    const int nsegs_cta = (nchunks + kChunksPerSeg - 1) / kChunksPerSeg;
    const int nstages = (nchunks + 1) / 2;
    uint8_t *hdr = smem + C::kOffHdr;
    prefetch_tmap(tmap);

    if constexpr (C::kQ8) {
        mbar_arrive(b.hdr);  // a Q8 copy has no segment headers
    } else {
        const uint32_t hbytes = (uint32_t)nsegs_cta * kSegHdrBytes;
        mbar_arrive_expect_tx(b.hdr, hbytes);
        bulk_g2s(hdr, p.blob + p.off_seg + (uint64_t)(tile * p.segs + s0) * kSegHdrBytes, hbytes, b.hdr);
    }
    bool hdr_ready = false;
    int issued = 0, seg_issued = 0;
    bool failed = false;

    for (int st = 0; st < nstages; ++st) {
        const int chunk = c0 + 2 * st;
        // the stage's packed chunks first: they need nothing from the header
        const int slot = st % C::kStages;
        if (st >= C::kStages &&
            !mbar_wait(b.wempty + slot, (uint32_t)(st / C::kStages - 1) & 1u, deadline)) {
            failed = true;
            break;
        }
        const int nch = min(2, c1 - chunk);
        mbar_arrive_expect_tx(b.wfull + slot, (uint32_t)(nch * C::kChunkB));
        bulk_g2s(smem + C::kOffW + slot * C::kWBytes,
                 p.blob + p.off_w + (uint64_t)(tile * p.chunks + chunk) * C::kChunkB, (uint32_t)(nch * C::kChunkB),
                 b.wfull + slot);
        issued = st + 1;
        if ((chunk & (kChunksPerSeg - 1)) == 0) {
            // a segment starts: its x tile (no header needed), then its escape
            // bytes; the one arrival comes last so the phase cannot complete early
            const int ls = chunk / kChunksPerSeg - s0;
            const int sslot = ls & 1;
            if (ls >= 2 && !mbar_wait(b.sempty + sslot, (uint32_t)((ls >> 1) - 1) & 1u, deadline)) {
                failed = true;
                break;
            }
            mbar_expect_tx(b.sfull + sslot, (uint32_t)C::kXBytes);
            uint8_t *xs = smem + C::kOffX + sslot * C::kXBytes;
#pragma unroll
            for (int bx = 0; bx < 4; ++bx)
                tma_load_2d(xs + bx * C::kXBoxBytes, tmap, chunk * kChunkK + bx * 64, 0, b.sfull + sslot);
            seg_issued = ls + 1;
            if constexpr (!C::kQ8) {
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
                    bulk_g2s(smem + C::kOffEsc + sslot * C::kEscCap, p.blob + p.off_esc + src0, ebytes,
                             b.sfull + sslot);
                }
            }
            mbar_arrive(b.sfull + sslot);
        }
        if (*abort_flag) break;
    }
    if (failed) raise_timeout(p.status, abort_flag);
    if (*abort_flag) {
        // let every copy still in flight land before the CTA can exit
        const uint64_t drain_deadline = globaltimer_ns() + 1000000000ull;
        for (int st = max(0, issued - C::kStages); st < issued; ++st)
            mbar_wait(b.wfull + st % C::kStages, (uint32_t)(st / C::kStages) & 1u, drain_deadline);
        for (int ls = max(0, seg_issued - 2); ls < seg_issued; ++ls)
            mbar_wait(b.sfull + (ls & 1), (uint32_t)(ls >> 1) & 1u, drain_deadline);
        mbar_wait(b.hdr, 0, drain_deadline);
    }
}

// ------------------------------------------------------------------ MMA issuer
// A chunk of 32 columns is two MMAs of K = 16.  B (x) sits in the segment's
// x tile: four 128-byte-swizzled boxes of 64 columns, K-major, 8-row atoms of
// 1024 B; columns 16u..16u+15 of a box start 32u bytes into it.
template <class C>
__device__ void gemm_mma(const GemmParams &p, uint8_t *smem, const Bars &b, volatile uint32_t *abort_flag,
                         uint32_t tmem_base, int c0, int nchunks, uint64_t deadline) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, C::kNtok);
    const int nstages = (nchunks + 1) / 2;
    bool failed = false;
    uint32_t xs = 0;
    for (int st = 0; st < nstages; ++st) {
        const int chunk0 = c0 + 2 * st;
        const int jj0 = chunk0 & (kChunksPerSeg - 1);
        const int ls = st / (kChunksPerSeg / 2);
        const int nch = min(2, c0 + nchunks - chunk0);
        if (jj0 == 0) {
            if (!mbar_wait(b.sfull + (ls & 1), (uint32_t)(ls >> 1) & 1u, deadline)) { failed = true; break; }
            xs = smem_u32(smem + C::kOffX + (ls & 1) * C::kXBytes);
        }
        const int aslot = st % C::kASlots;
        if (!mbar_wait(b.afull + aslot, (uint32_t)(st / C::kASlots) & 1u, deadline)) { failed = true; break; }
        tc_fence_after();
        for (int e = 0; e < nch; ++e) {
            const int jj = jj0 + e;
            const uint32_t xbox = xs + (uint32_t)(jj >> 1) * C::kXBoxBytes + (uint32_t)(jj & 1) * 64u;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const uint64_t bdesc = smem_desc(xbox + (uint32_t)kk * 32u, 16u, 1024u, 2u);
                const uint32_t acc = (st > 0 || e > 0 || kk > 0) ? 1u : 0u;
                if constexpr (C::kASmem) {
                    // K-major, no swizzle: 8x16-byte core matrices, 128 B apart
                    // along K, 512 B apart along rows; MMA kk starts 256 B in.
                    const uint32_t as = smem_u32(smem + C::kOffA + aslot * C::kASlotBytes + e * C::kAChunkBytes) +
                                        (uint32_t)kk * 256u;
                    mma_smem_a(tmem_base + C::kDCol, smem_desc(as, 128u, 512u, 0u), bdesc, idesc, acc);
                } else {
                    // slot columns: [k-half kk][chunk e] x 8 (one decode warp's 16 columns are contiguous)
                    mma_tmem_a(tmem_base + C::kDCol,
                               tmem_base + C::kACol + (uint32_t)(32 * aslot + 16 * kk + 8 * e), bdesc, idesc, acc);
                }
            }
        }
        mma_commit(b.aempty + aslot);
        if (jj0 + nch == kChunksPerSeg || st == nstages - 1) mma_commit(b.sempty + (ls & 1));
        if (*abort_flag) break;
    }
    if (failed) raise_timeout(p.status, abort_flag);
    mma_commit(b.accum);  // also fires when nothing was issued
    // before TMEM can be freed every issued MMA must have completed
    mma_commit(b.drain);
    mbar_wait(b.drain, 0, globaltimer_ns() + 1000000000ull);
}

// ------------------------------------------------------------------ decoders
// One chunk's half-row: decode 16 weights of row r, columns 16h..16h+15.
__device__ __forceinline__ void decode_half_chunk(const Table &T, const uint4 &sb, const uint4 &codes, int h,
                                                  bool has_escapes, const uint8_t *&run, uint32_t (&out)[8]) {
    uint32_t E[4];
    if (has_escapes)
        run += decode_exponents_half_esc(T, codes, h, run, E);
    else
        decode_exponents_half(T, h ? codes.z : codes.x, h ? codes.w : codes.y, E);
    assemble_half(sb, E, out);
}

template <class C>
__device__ void gemm_decode(const GemmParams &p, uint8_t *smem, const Bars &b, volatile uint32_t *abort_flag,
                            uint32_t tmem_base, int s0, int c0, int c1, uint64_t deadline) {
    const int warp = threadIdx.x >> 5;
    const int q = warp & 3;       // TMEM lane quarter = rows 32q..32q+31
    const int h = warp >> 2;      // columns 16h..16h+15 of each chunk
    const int lane = threadIdx.x & 31;
    const int r = 32 * q + lane;  // row in the tile
    const int nchunks = c1 - c0;
    const int nstages = (nchunks + 1) / 2;
    const uint8_t *hdr = smem + C::kOffHdr;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    // this thread's S bytes (half h of its row) in weight stage 0; codes are
    // c_off further on
    const uint32_t s_row = smem_u32(smem + C::kOffW) + (uint32_t)(h * kSlabBytes + 16 * r);
    const uint32_t c_off = (uint32_t)((2 - h) * kSlabBytes);

    if (!warp_wait(b.hdr, 0, deadline)) {
        if (lane == 0) raise_timeout(p.status, abort_flag);
        return;
    }
    Table T{};
    uint32_t mask_q = 0;
    const uint8_t *run = nullptr;
    // The handshake for stage st (wait for its TMEM stores, tell the MMA warp)
    // is made one stage later, so that the store latency overlaps the next
    // stage's decode.
    int pend_slot = -1;
    bool pend_seg_end = false;
    int pend_ls = 0;
    for (int st = 0; st < nstages; ++st) {
        const int chunk0 = c0 + 2 * st;
        const int jj0 = chunk0 & (kChunksPerSeg - 1);
        const int ls = st / (kChunksPerSeg / 2);
        const int nch = min(2, c1 - chunk0);
        if (!C::kQ8 && jj0 == 0) {
            const uint8_t *hp = hdr + (chunk0 / kChunksPerSeg - s0) * kSegHdrBytes;
            T = make_table(*reinterpret_cast<const uint4 *>(hp));
            const uint4 meta = *reinterpret_cast<const uint4 *>(hp + 16);
            const uint32_t qc0 = meta.y & 0xFFFFu, qc1 = meta.y >> 16, qc2 = meta.z & 0xFFFFu;
            const uint32_t qoff = (q > 0 ? qc0 : 0u) + (q > 1 ? qc1 : 0u) + (q > 2 ? qc2 : 0u);
            mask_q = (meta.w >> (8 * q)) & 0xFFu;
            if (!warp_wait(b.sfull + (ls & 1), (uint32_t)(ls >> 1) & 1u, deadline)) {
                if (lane == 0) raise_timeout(p.status, abort_flag);
                return;
            }
            if (escapes_staged<C>(seg_escape_total(meta)))
                run = smem + C::kOffEsc + (ls & 1) * C::kEscCap + (meta.x & 15u) + qoff;
            else
                run = p.blob + p.off_esc + meta.x + qoff;
        }
        const int slot = st % C::kStages;
        if (!warp_wait(b.wfull + slot, (uint32_t)(st / C::kStages) & 1u, deadline)) {
            if (lane == 0) raise_timeout(p.status, abort_flag);
            return;
        }
        const uint32_t sa = s_row + (uint32_t)(slot * C::kWBytes);
        const uint4 sb0 = lds128(sa);
        const uint4 cd0 = C::kQ8 ? make_uint4(0, 0, 0, 0) : lds128(sa + c_off);
        uint4 sb1 = make_uint4(0, 0, 0, 0), cd1 = make_uint4(0, 0, 0, 0);
        if (nch == 2) {
            sb1 = lds128(sa + C::kChunkB);
            if (!C::kQ8) cd1 = lds128(sa + C::kChunkB + c_off);
        }
        warp_arrive(b.wempty + slot);  // this warp is done with the stage's bytes

        uint32_t out0[8], out1[8];
        if constexpr (C::kQ8) {
            // 8-bit copy: 16 int8 per chunk half, exact in BF16
            q8_half(sb0, out0);
            q8_half(sb1, out1);  // a short last stage leaves these columns unread
        } else if (nch == 2 && ((mask_q >> jj0) & 3u) == 0) {
            // common case, decided once per stage for the whole warp: two
            // chunks without escapes
            uint32_t E[4];
            decode_exponents_half(T, h ? cd0.z : cd0.x, h ? cd0.w : cd0.y, E);
            assemble_half(sb0, E, out0);
            decode_exponents_half(T, h ? cd1.z : cd1.x, h ? cd1.w : cd1.y, E);
            assemble_half(sb1, E, out1);
        } else {
            decode_half_chunk(T, sb0, cd0, h, (mask_q >> jj0) & 1u, run, out0);
            if (nch == 2) {
                decode_half_chunk(T, sb1, cd1, h, (mask_q >> (jj0 + 1)) & 1u, run, out1);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) out1[i] = 0u;
            }
        }

        if constexpr (!C::kASmem) {
            if (pend_slot >= 0) {
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(b.afull + pend_slot);
                    if (pend_seg_end) mbar_arrive(b.sempty + (pend_ls & 1));
                }
                pend_slot = -1;
            }
        }
        const int aslot = st % C::kASlots;
        if (st >= C::kASlots &&
            !warp_wait(b.aempty + aslot, (uint32_t)(st / C::kASlots - 1) & 1u, deadline)) {
            if (lane == 0) raise_timeout(p.status, abort_flag);
            return;
        }
        if constexpr (C::kASmem) {
            uint8_t *ap = smem + C::kOffA + aslot * C::kASlotBytes + (r >> 3) * 512 + (r & 7) * 16 + h * 256;
#pragma unroll
            for (int g = 0; g < 2; ++g)
                *reinterpret_cast<uint4 *>(ap + g * 128) =
                    make_uint4(out0[4 * g], out0[4 * g + 1], out0[4 * g + 2], out0[4 * g + 3]);
            if (nch == 2) {
#pragma unroll
                for (int g = 0; g < 2; ++g)
                    *reinterpret_cast<uint4 *>(ap + C::kAChunkBytes + g * 128) =
                        make_uint4(out1[4 * g], out1[4 * g + 1], out1[4 * g + 2], out1[4 * g + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(b.afull + aslot);
                if (jj0 + nch == kChunksPerSeg || st == nstages - 1) mbar_arrive(b.sempty + (ls & 1));
            }
        } else {
            tc_fence_after();
            const uint32_t ta = tmem_base + lane_base + (uint32_t)(C::kACol + 32 * aslot + 16 * h);
            uint32_t v[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                v[i] = out0[i];
                v[8 + i] = out1[i];  // a short last stage leaves these columns unread
            }
            tmem_st16(ta, v);
            pend_slot = aslot;
            pend_seg_end = (jj0 + nch == kChunksPerSeg || st == nstages - 1);
            pend_ls = ls;
        }
    }
    if constexpr (!C::kASmem) {
        if (pend_slot >= 0) {
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(b.afull + pend_slot);
                if (pend_seg_end) mbar_arrive(b.sempty + (pend_ls & 1));
            }
        }
    }
}

// ------------------------------------------------------------------ epilogue
// The last CTA of a tile sums the tile's split partials in ascending split
// order (fixed, so results repeat run to run) and stores y.  The M x 128
// outputs are spread over the CTA's decode threads; a thread keeps several
// loads in flight: eight splits of one output when it has one or two outputs,
// else kUnroll splits of kBatch outputs.
template <int kThreads, int kBatch, int kUnroll>
__device__ __forceinline__ void reduce_splits(const GemmParams &p, int64_t tile, int t) {
    static_assert(kThreads % kTileRows == 0, "outputs of one thread share a row");
    const int total = p.M * kTileRows;
    const int64_t sstride = (int64_t)p.M * p.Npad;
    const float *base = p.partials + tile * kTileRows;
    if (total <= 2 * kThreads) {
        // total is a multiple of 128, so a warp's lanes leave this loop together
        for (int o = t; o < total; o += kThreads) {
            const int m = o / kTileRows, rr = o % kTileRows;
            const bool valid = tile * kTileRows + rr < p.N;
            const float *src = base + (int64_t)m * p.Npad + (valid ? rr : 0);
            float s = 0.0f;
            int sp = 0;
            for (; sp + 8 <= p.splits; sp += 8) {
                float v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = __ldcg(src + (sp + u) * sstride);
#pragma unroll
                for (int u = 0; u < 8; ++u) s += v[u];
            }
            for (; sp < p.splits; ++sp) s += __ldcg(src + sp * sstride);
            if (p.scales != nullptr) s *= p.scales[tile * kTileRows + rr];
            if (p.y != nullptr && valid) p.y[(int64_t)m * p.N + tile * kTileRows + rr] = bf16_bits_rn(s);
            if (p.amax != nullptr)
                argmax_warp(p.amax + m, valid ? argmax_key(s, (uint32_t)(tile * kTileRows + rr)) : 0ull);
        }
        return;
    }
    for (int o0 = t; o0 < total; o0 += kBatch * kThreads) {
        float s[kBatch];
        uint32_t ok = 0;  // bit b: output o0 + b * kThreads exists
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int o = o0 + b * kThreads;
            if (o < total && tile * kTileRows + o % kTileRows < p.N) ok |= 1u << b;
            s[b] = 0.0f;
        }
        // outputs b and b + 1 are kThreads / 128 tokens apart, same row
        const float *src = base + (int64_t)(o0 / kTileRows) * p.Npad + o0 % kTileRows;
        constexpr int kTokStep = kThreads / kTileRows;
        int sp = 0;
        for (; sp + kUnroll <= p.splits; sp += kUnroll) {
            float v[kUnroll][kBatch];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
#pragma unroll
                for (int b = 0; b < kBatch; ++b)
                    v[u][b] = (ok >> b) & 1u
                                  ? __ldcg(src + (sp + u) * sstride + (int64_t)(b * kTokStep) * p.Npad)
                                  : 0.0f;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
#pragma unroll
                for (int b = 0; b < kBatch; ++b) s[b] += v[u][b];
        }
        for (; sp < p.splits; ++sp) {
#pragma unroll
            for (int b = 0; b < kBatch; ++b)
                s[b] += (ok >> b) & 1u ? __ldcg(src + sp * sstride + (int64_t)(b * kTokStep) * p.Npad) : 0.0f;
        }
        if (p.scales != nullptr) {
            const float sc = p.scales[tile * kTileRows + o0 % kTileRows];  // one row for all b
#pragma unroll
            for (int b = 0; b < kBatch; ++b) s[b] *= sc;
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int o = o0 + b * kThreads;
            if (p.y != nullptr && ((ok >> b) & 1u))
                p.y[(int64_t)(o / kTileRows) * p.N + tile * kTileRows + o % kTileRows] = bf16_bits_rn(s[b]);
            // o < total is the same for the 32 lanes of a warp
            if (p.amax != nullptr && o < total)
                argmax_warp(p.amax + o / kTileRows,
                            ((ok >> b) & 1u) ? argmax_key(s[b], (uint32_t)(tile * kTileRows + o % kTileRows)) : 0ull);
        }
    }
}

// D (fp32, TMEM lane = weight row, column = token) -> y, or -> partials and
// the last CTA of the tile sums the partials in split order.
template <class C>
__device__ void gemm_epilogue(const GemmParams &p, const Bars &b, volatile uint32_t *abort_flag,
                              volatile uint32_t *last_flag, uint32_t tmem_base, int64_t tile, int split,
                              uint64_t deadline) {
    const int warp = threadIdx.x >> 5;
    const int q = warp & 3;
    const int h = warp >> 2;
    const int lane = threadIdx.x & 31;
    constexpr int kHalf = C::kNtok / 2;  // this warp's tokens: h*kHalf .. h*kHalf + kHalf - 1
    const int m0 = h * kHalf;
    if (!warp_wait(b.accum, 0, deadline)) {
        if (lane == 0) raise_timeout(p.status, abort_flag);
        return;
    }
    tc_fence_after();
    float acc[kHalf];
    {
        const uint32_t ta = tmem_base + ((uint32_t)(32 * q) << 16) + C::kDCol + (uint32_t)m0;
        if constexpr (kHalf == 8) {
            uint32_t v[8];
            tmem_ld8(ta, v);
            tmem_wait_ld();
#pragma unroll
            for (int m = 0; m < 8; ++m) acc[m] = __uint_as_float(v[m]);
        } else {
            uint32_t v[16];
            tmem_ld16(ta, v);
            tmem_wait_ld();
#pragma unroll
            for (int m = 0; m < 16; ++m) acc[m] = __uint_as_float(v[m]);
        }
    }
    const int64_t n = tile * kTileRows + 32 * q + lane;
    if (p.splits == 1) {
        if (p.scales != nullptr) {
            const float sc = p.scales[n];  // rows past N have scale 0
#pragma unroll
            for (int m = 0; m < kHalf; ++m) acc[m] *= sc;
        }
        if (p.y != nullptr && n < p.N) {
#pragma unroll
            for (int m = 0; m < kHalf; ++m)
                if (m0 + m < p.M) p.y[(int64_t)(m0 + m) * p.N + n] = bf16_bits_rn(acc[m]);
        }
        if (p.amax != nullptr) {
#pragma unroll
            for (int m = 0; m < kHalf; ++m)
                if (m0 + m < p.M) argmax_warp(p.amax + m0 + m, n < p.N ? argmax_key(acc[m], (uint32_t)n) : 0ull);
        }
        return;
    }
    float *part = p.partials + (int64_t)split * p.M * p.Npad + n;
#pragma unroll
    for (int m = 0; m < kHalf; ++m)
        if (m0 + m < p.M) __stcg(part + (int64_t)(m0 + m) * p.Npad, acc[m]);
    // the decode warps meet on mbarriers (bounded waits, no bar.sync that
    // a warp which gave up could leave the others stuck in); the mbarrier
    // arrive/wait pair orders this CTA's partial stores before thread 0's
    // fence, which publishes them all with the counter increment
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
    reduce_splits<C::kDecWarps * 32, 8, C::kNtok == 16 ? 3 : 4>(p, tile, (int)threadIdx.x);
    if (threadIdx.x == 0) p.counters[tile] = 0u;  // ready for the next call
}

// ------------------------------------------------------------------ kernel
template <int NTOK, int STAGES, bool A_SMEM, bool Q8 = false>
__global__ void __launch_bounds__(320, NTOK == 16 ? 3 : 2)
    w12_gemm_tc_kernel(const __grid_constant__ GemmGroup grp, const __grid_constant__ CUtensorMap tmap_x) {
    using C = GemmCfg<NTOK, STAGES, A_SMEM, Q8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBars);
    Bars b;
    b.wfull = bars;
    b.wempty = b.wfull + STAGES;
    b.sfull = b.wempty + STAGES;
    b.sempty = b.sfull + C::kSegSlots;
    b.afull = b.sempty + C::kSegSlots;
    b.aempty = b.afull + C::kASlots;
    b.hdr = b.aempty + C::kASlots;
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
            mbar_init(b.sempty + i, C::kDecWarps + 1);
        }
        for (int i = 0; i < C::kASlots; ++i) {
            mbar_init(b.afull + i, C::kDecWarps);
            mbar_init(b.aempty + i, 1);
        }
        mbar_init(b.hdr, 1);
        mbar_init(b.accum, 1);
        mbar_init(b.drain, 1);
        mbar_init(b.epi_in, C::kDecWarps);
        mbar_init(b.epi_out, 1);
        *abort_flag = 0u;
        *last_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0) pdl_launch_dependents();
    if (warp == 8 && (threadIdx.x & 31) == 0) {
        uint32_t budget = kPrefetchBytes;
        prefetch_cta_weights<C::kChunkB, !Q8>(p, tile, s0, c0, c1, budget);
    }
    pdl_wait();

    if (warp == 8) {
        if ((threadIdx.x & 31) == 0) gemm_producer<C>(p, &tmap_x, smem, b, abort_flag, tile, s0, c0, c1, deadline);
    } else if (warp == 9) {
        if ((threadIdx.x & 31) == 0) gemm_mma<C>(p, smem, b, abort_flag, tmem_base, c0, c1 - c0, deadline);
        __syncwarp();
    } else {
        gemm_decode<C>(p, smem, b, abort_flag, tmem_base, s0, c0, c1, deadline);
        gemm_epilogue<C>(p, b, abort_flag, last_flag, tmem_base, tile, split, deadline);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem_base, C::kTmemCols);
}

}  // namespace dev
}  // namespace w12
