// W12 v1 encoder on the GPU: the same canonical bytes as the host encoder
// (format: include/w12.h) for weights already resident in device memory.
// Lossless and bit-exact ("StargazerX0/SpecPilot", §What it is; "SpecPilot",
// §Differentiation), ~12 bits per weight ("SpecPilot: an agent doubled
// speculative decoding speed, and the 10.87x needs context", §The mechanisms
// it found).
//
//   plan    one CTA per segment (128 rows x 256 columns, grid-stride): one
//           exponent histogram per (quarter, chunk) block in shared memory;
//           their sum ranks the 15 most frequent exponents (count, then the
//           smaller exponent) and the slot rule places them; the escape count
//           of each block is the mass of its histogram outside the table.
//           Output: a 32-byte record per segment (table, quarter counts, chunk
//           mask, total).
//   scan    one CTA: exclusive prefix of the segment totals in blob order
//           (tile, then segment) -> each segment's first escape offset.
//   write   one CTA of 128 threads per segment (grid-stride), thread = row,
//           warp = quarter: S bytes and codes of each chunk, escape bytes
//           placed by a warp scan (order: quarter, chunk, row, column).
//   header  the 256-byte header and the zero padding between the planes.
// Every write into the blob is bounded by the caller's capacity; an overflow
// or an escape count above 2^32-1 is recorded in the status word.
#pragma once

#include <cstdint>

#include "w12_format.hpp"

namespace w12 {
namespace dev {

struct EncodeParams {
    const uint16_t *w;    // N x K row-major BF16 bit patterns
    int64_t N, K, Kp, tiles, chunks, segs;
    int vec;              // rows 16-byte aligned: w 16-byte aligned and K % 8 == 0
    uint8_t *plan;        // [tiles * segs] x 32 B records
    uint64_t *base;       // [tiles * segs] first escape offset
    uint64_t *n_esc;      // total escape count
    uint8_t *blob;        // output, blob_bytes long
    uint64_t blob_bytes;
    uint64_t off_seg, off_w, off_esc;
    uint32_t *status;
};

constexpr uint32_t kStatusEncodeOverflow = 16u;   // blob buffer shorter than the encoding
constexpr uint32_t kStatusEncodeEscapes = 32u;    // more than 2^32-1 escapes

// Plan record layout (32 bytes).
constexpr int kRecTable = 0, kRecQcount = 16, kRecMask = 24, kRecTotal = 28;

__device__ __forceinline__ uint16_t enc_weight(const EncodeParams &p, int64_t n, int64_t k) {
    return (n < p.N && k < p.K) ? p.w[n * p.K + k] : (uint16_t)0;
}

__device__ __forceinline__ uint32_t exp_of(uint32_t b) { return (b >> 7) & 0xFFu; }

// Code of exponent e under table t: the first slot 0-14 holding e, else 15.
__device__ __forceinline__ uint32_t code_for(const uint8_t *t, uint32_t e) {
    uint32_t c = 15;
#pragma unroll
    for (int s = 14; s >= 0; --s)
        if (t[s] == e) c = (uint32_t)s;
    return c;
}

__global__ void __launch_bounds__(256) w12_encode_plan_kernel(const __grid_constant__ EncodeParams p) {
    __shared__ uint32_t sub[32][256];   // [quarter * 8 + chunk][exponent]
    __shared__ uint32_t hist[256];
    __shared__ uint8_t is_esc[256];
    __shared__ int16_t slot[16];
    __shared__ uint8_t table[16];
    __shared__ uint32_t esc[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t nseg = p.tiles * p.segs;
    for (int64_t sidx = blockIdx.x; sidx < nseg; sidx += gridDim.x) {
        const int64_t tile = sidx / p.segs;
        const int64_t seg = sidx % p.segs;
        __syncthreads();  // the previous segment is done with the shared arrays
        for (int i = tid; i < 32 * 256; i += 256) (&sub[0][0])[i] = 0;
        if (tid < 16) slot[tid] = -1;
        __syncthreads();

        const int64_t k0 = seg * kSegK;
        const int64_t n0 = tile * kTileRows;
        const int width = (int)(p.Kp - k0 < kSegK ? p.Kp - k0 : kSegK);
        if (p.vec && n0 + kTileRows <= p.N && k0 + kSegK <= p.K) {
            // full segment, 8 weights per load; a warp covers one row
            for (int i = tid; i < kTileRows * kSegK / 8; i += 256) {
                const int r = i >> 5, c8 = (i & 31) * 8;
                const uint4 v = *reinterpret_cast<const uint4 *>(p.w + (n0 + r) * p.K + k0 + c8);
                uint32_t *h = sub[(r / kQuarterRows) * 8 + c8 / kChunkK];
                const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    atomicAdd(&h[exp_of(u[j])], 1u);
                    atomicAdd(&h[exp_of(u[j] >> 16)], 1u);
                }
            }
        } else {
            for (int i = tid; i < kTileRows * width; i += 256) {
                const int r = i / width, c = i % width;
                atomicAdd(&sub[(r / kQuarterRows) * 8 + c / kChunkK][exp_of(enc_weight(p, n0 + r, k0 + c))], 1u);
            }
        }
        __syncthreads();
        {
            uint32_t s = 0;
#pragma unroll 8
            for (int b = 0; b < 32; ++b) s += sub[b][tid];
            hist[tid] = s;
        }
        __syncthreads();

        if (warp == 0) {
            // lane l holds exponents 8l .. 8l+7; key = count * 256 + (255 - e):
            // the larger count wins, then the smaller exponent
            uint64_t key[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = lane * 8 + i;
                key[i] = hist[e] ? (((uint64_t)hist[e] << 8) | (uint64_t)(255 - e)) : 0ull;
            }
            uint32_t chosen = 0;  // bit i: exponent 8 * lane + i is in the table
            for (int round = 0; round < 15; ++round) {
                uint64_t best = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (!((chosen >> i) & 1u) && key[i] > best) best = key[i];
#pragma unroll
                for (int off = 16; off; off >>= 1) {
                    const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, best, off);
                    best = o > best ? o : best;
                }
                if (best == 0) break;
                const int e = 255 - (int)(best & 0xFF);
                if ((e >> 3) == lane) chosen |= 1u << (e & 7);
            }
            // slot rule: the chosen exponents below 128 (lanes 0-15) and from 128
            // up (lanes 16-31), each group ascending, are laid along the visit
            // order 7,0,8,1,...,6,14 (position v -> slot 7 + v/2 for even v,
            // (v-1)/2 for odd v); the group with an odd count goes first (the low
            // group if both are odd, or if neither is) and, when both counts are
            // even, the walk starts at its second position so that slot 7 stays
            // free for the escape pairing
            const uint32_t cnt = __popc(chosen);
            uint32_t incl = cnt;
#pragma unroll
            for (int d = 1; d < 16; d <<= 1) {
                const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if ((lane & 15) >= d) incl += o;
            }
            const uint32_t nlow = __shfl_sync(0xFFFFFFFFu, incl, 15);
            const uint32_t nhigh = __shfl_sync(0xFFFFFFFFu, incl, 31);
            const bool low_first = (nlow & 1u) || !(nhigh & 1u);
            const uint32_t start = ((nlow & 1u) || (nhigh & 1u)) ? 0u : 1u;
            const bool high_lane = lane >= 16;
            uint32_t pos = start + (incl - cnt);
            if (high_lane == low_first) pos += high_lane ? nlow : nhigh;
            for (int i = 0; i < 8; ++i) {
                if ((chosen >> i) & 1u) {
                    const uint32_t v = pos++;
                    slot[(v & 1u) ? (v - 1) >> 1 : 7 + (v >> 1)] = (int16_t)(lane * 8 + i);
                }
            }
            __syncwarp();
            if (lane < 15) {
                int16_t v = slot[lane];
                if (v < 0) {
                    const int partner = lane == 7 ? 15 : (lane ^ 8);
                    v = slot[partner] >= 0 ? slot[partner] : (int16_t)0;
                }
                table[lane] = (uint8_t)v;
            } else if (lane == 15) {
                table[15] = 0;
            }
        }
        __syncthreads();
        is_esc[tid] = code_for(table, (uint32_t)tid) == 15 ? 1 : 0;
        __syncthreads();
#pragma unroll
        for (int b = warp * 4; b < warp * 4 + 4; ++b) {
            uint32_t s = 0;
#pragma unroll
            for (int e = lane; e < 256; e += 32) s += is_esc[e] ? sub[b][e] : 0u;
#pragma unroll
            for (int off = 16; off; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
            if (lane == 0) esc[b] = s;
        }
        __syncthreads();
        if (tid == 0) {
            uint8_t *rec = p.plan + (uint64_t)sidx * 32;
            uint32_t mask = 0, total = 0;
            for (int c = 0; c < 16; ++c) rec[kRecTable + c] = table[c];
            for (int q = 0; q < 4; ++q) {
                uint32_t qc = 0;
                for (int j = 0; j < 8; ++j) {
                    qc += esc[q * 8 + j];
                    if (esc[q * 8 + j]) mask |= 1u << (8 * q + j);
                }
                rec[kRecQcount + 2 * q] = (uint8_t)qc;
                rec[kRecQcount + 2 * q + 1] = (uint8_t)(qc >> 8);
                total += qc;
            }
            *reinterpret_cast<uint32_t *>(rec + kRecMask) = mask;
            *reinterpret_cast<uint32_t *>(rec + kRecTotal) = total;
        }
    }
}

// Exclusive prefix of the segment totals, one CTA of 1024 threads.
__global__ void __launch_bounds__(1024) w12_encode_scan_kernel(const __grid_constant__ EncodeParams p) {
    __shared__ uint64_t warp_incl[32];
    __shared__ uint64_t carry;
    const int64_t nseg = p.tiles * p.segs;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int64_t start = 0; start < nseg; start += 1024) {
        const int64_t i = start + tid;
        const uint64_t v = i < nseg ? *reinterpret_cast<const uint32_t *>(p.plan + i * 32 + kRecTotal) : 0ull;
        uint64_t incl = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint64_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= d) incl += o;
        }
        if (lane == 31) warp_incl[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            uint64_t s = warp_incl[lane];
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint64_t o = __shfl_up_sync(0xFFFFFFFFu, s, d);
                if (lane >= d) s += o;
            }
            warp_incl[lane] = s;
        }
        __syncthreads();
        const uint64_t before = carry + (warp ? warp_incl[warp - 1] : 0ull) + (incl - v);
        if (i < nseg) p.base[i] = before;
        __syncthreads();
        if (tid == 1023) carry = before + v;
        __syncthreads();
    }
    if (tid == 0) {
        *p.n_esc = carry;
        if (p.blob != nullptr && carry > 0xFFFFFFFFull) atomicOr(p.status, kStatusEncodeEscapes);
    }
}

__global__ void __launch_bounds__(128) w12_encode_write_kernel(const __grid_constant__ EncodeParams p) {
    __shared__ uint8_t rec[32];
    __shared__ uint8_t code_of[256];
    const int r = threadIdx.x, q = r >> 5, lane = r & 31;
    const int64_t nseg = p.tiles * p.segs;
    for (int64_t sidx = blockIdx.x; sidx < nseg; sidx += gridDim.x) {
        const int64_t tile = sidx / p.segs;
        const int64_t seg = sidx % p.segs;
        __syncthreads();  // the previous segment is done with rec and code_of
        if (r < 32) rec[r] = p.plan[sidx * 32 + r];
        __syncthreads();
        code_of[r] = (uint8_t)code_for(rec + kRecTable, (uint32_t)r);
        code_of[r + 128] = (uint8_t)code_for(rec + kRecTable, (uint32_t)r + 128);
        const uint64_t base = p.base[sidx];
        if (r == 0) {
            const uint64_t at = p.off_seg + (uint64_t)sidx * kSegHdrBytes;
            if (at + kSegHdrBytes <= p.blob_bytes) {
                uint8_t *h = p.blob + at;
                for (int i = 0; i < 16; ++i) h[i] = rec[kRecTable + i];
                for (int i = 0; i < 4; ++i) h[16 + i] = (uint8_t)(base >> (8 * i));
                for (int i = 0; i < 8; ++i) h[20 + i] = rec[kRecQcount + i];
                for (int i = 0; i < 4; ++i) h[28 + i] = rec[kRecMask + i];
            } else {
                atomicOr(p.status, kStatusEncodeOverflow);
            }
        }
        __syncthreads();
        uint64_t run = base;  // this quarter's next escape offset
        for (int qq = 0; qq < q; ++qq)
            run += (uint32_t)rec[kRecQcount + 2 * qq] | ((uint32_t)rec[kRecQcount + 2 * qq + 1] << 8);
        const int64_t n = tile * kTileRows + r;
        const int64_t jbeg = seg * kChunksPerSeg;
        const int64_t jend = jbeg + kChunksPerSeg < p.chunks ? jbeg + kChunksPerSeg : p.chunks;
        for (int64_t j = jbeg; j < jend; ++j) {
            const int64_t k0 = j * kChunkK;
            uint32_t u[16];  // 32 weights, two per word, column order
            if (p.vec && n < p.N && k0 + kChunkK <= p.K) {
                const uint4 *src = reinterpret_cast<const uint4 *>(p.w + n * p.K + k0);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 v = src[i];
                    u[4 * i] = v.x, u[4 * i + 1] = v.y, u[4 * i + 2] = v.z, u[4 * i + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    u[i] = (uint32_t)enc_weight(p, n, k0 + 2 * i) | ((uint32_t)enc_weight(p, n, k0 + 2 * i + 1) << 16);
            }
            uint32_t sw[8] = {0, 0, 0, 0, 0, 0, 0, 0}, cw[4] = {0, 0, 0, 0};
            uint32_t cnt = 0;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                // columns 2i and 2i+1 carry each other's sign
                const uint32_t a = u[i] & 0xFFFFu, b = u[i] >> 16;
                const uint32_t sa = ((a & 0x7Fu) << 1) | (b >> 15);
                const uint32_t sb = ((b & 0x7Fu) << 1) | (a >> 15);
                sw[i >> 1] |= (sa | (sb << 8)) << (16 * (i & 1));
                const uint32_t ca = code_of[exp_of(a)], cb = code_of[exp_of(b)];
                cw[i >> 2] |= (ca | (cb << 4)) << (8 * (i & 3));
                cnt += (ca == 15) + (cb == 15);
            }
            const uint64_t at = p.off_w + (uint64_t)(tile * p.chunks + j) * kChunkBytes;
            if (at + kChunkBytes <= p.blob_bytes) {
                uint8_t *cp = p.blob + at;
                *reinterpret_cast<uint4 *>(cp + 16 * r) = make_uint4(sw[0], sw[1], sw[2], sw[3]);
                *reinterpret_cast<uint4 *>(cp + kSlabBytes + 16 * r) = make_uint4(sw[4], sw[5], sw[6], sw[7]);
                *reinterpret_cast<uint4 *>(cp + 2 * kSlabBytes + 16 * r) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
            } else {
                atomicOr(p.status, kStatusEncodeOverflow);
            }
            uint32_t incl = cnt;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if (lane >= d) incl += o;
            }
            const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
            if (cnt) {
                uint64_t pos = p.off_esc + run + (incl - cnt);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const uint32_t b = (u[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
                    if (code_of[exp_of(b)] == 15) {
                        if (pos < p.blob_bytes) p.blob[pos] = (uint8_t)exp_of(b);
                        else atomicOr(p.status, kStatusEncodeOverflow);
                        ++pos;
                    }
                }
            }
            run += total;
        }
    }
}

__device__ __forceinline__ void put_le_dev(uint8_t *b, int off, uint64_t v, int n) {
    for (int i = 0; i < n; ++i) b[off + i] = (uint8_t)(v >> (8 * i));
}

// The header and the zero gaps; one CTA.
__global__ void __launch_bounds__(256) w12_encode_header_kernel(const __grid_constant__ EncodeParams p) {
    const uint64_t n_esc = *p.n_esc;
    const uint64_t bytes_esc = (n_esc + 15) / 16 * 16;
    const uint64_t total = (p.off_esc + bytes_esc + kPlaneAlign - 1) / kPlaneAlign * kPlaneAlign;
    const uint64_t bytes_seg = (uint64_t)kSegHdrBytes * (uint64_t)(p.tiles * p.segs);
    const uint64_t bytes_w = (uint64_t)kChunkBytes * (uint64_t)(p.tiles * p.chunks);
    if (total > p.blob_bytes) {
        if (threadIdx.x == 0) atomicOr(p.status, kStatusEncodeOverflow);
        return;
    }
    constexpr uint64_t kHeaderUsed = hdr::kTotal + 8;
    for (uint64_t i = kHeaderUsed + threadIdx.x; i < (uint64_t)kHeaderBytes; i += blockDim.x) p.blob[i] = 0;
    for (uint64_t i = p.off_seg + bytes_seg + threadIdx.x; i < p.off_w; i += blockDim.x) p.blob[i] = 0;
    for (uint64_t i = p.off_w + bytes_w + threadIdx.x; i < p.off_esc; i += blockDim.x) p.blob[i] = 0;
    for (uint64_t i = p.off_esc + n_esc + threadIdx.x; i < total; i += blockDim.x) p.blob[i] = 0;
    if (threadIdx.x != 0) return;
    uint8_t *b = p.blob;
    put_le_dev(b, hdr::kMagicOff, kMagic, 4);
    put_le_dev(b, hdr::kVersionOff, kVersion, 4);
    put_le_dev(b, hdr::kHeaderBytesOff, kHeaderBytes, 4);
    put_le_dev(b, hdr::kFlagsOff, 0, 4);
    put_le_dev(b, hdr::kN, (uint64_t)p.N, 8);
    put_le_dev(b, hdr::kK, (uint64_t)p.K, 8);
    put_le_dev(b, hdr::kNpad, (uint64_t)(p.tiles * kTileRows), 8);
    put_le_dev(b, hdr::kKpad, (uint64_t)p.Kp, 8);
    put_le_dev(b, hdr::kTileRowsOff, kTileRows, 4);
    put_le_dev(b, hdr::kChunkKOff, kChunkK, 4);
    put_le_dev(b, hdr::kSegKOff, kSegK, 4);
    put_le_dev(b, hdr::kQuarterOff, kQuarterRows, 4);
    put_le_dev(b, hdr::kTiles, (uint64_t)p.tiles, 8);
    put_le_dev(b, hdr::kChunks, (uint64_t)p.chunks, 8);
    put_le_dev(b, hdr::kSegs, (uint64_t)p.segs, 8);
    put_le_dev(b, hdr::kOffSeg, p.off_seg, 8);
    put_le_dev(b, hdr::kBytesSeg, bytes_seg, 8);
    put_le_dev(b, hdr::kOffW, p.off_w, 8);
    put_le_dev(b, hdr::kBytesW, bytes_w, 8);
    put_le_dev(b, hdr::kOffEsc, p.off_esc, 8);
    put_le_dev(b, hdr::kNEsc, n_esc, 8);
    put_le_dev(b, hdr::kBytesEsc, bytes_esc, 8);
    put_le_dev(b, hdr::kTotal, total, 8);
}

}  // namespace dev
}  // namespace w12
