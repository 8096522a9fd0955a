// W12 -> BF16 decode kernel: the bit-exact inverse of the encoder
// ("decodes bit-exactly": "StargazerX0/SpecPilot", §What it is; "lossless":
// "SpecPilot", §Differentiation).
//
// One CTA of 128 threads per (tile, segment); warp q owns quarter q (32 rows),
// each thread one row.  Per chunk a warp reads its 3 x 512 contiguous bytes
// with 16-byte loads and decodes in registers (same routine as the GEMM).  The
// 64 output bytes of each row are staged in shared memory and written back
// 8 rows x 64 bytes per warp instruction, so each store covers whole 32-byte
// sectors instead of 16 bytes in each of 32 rows.  Streams 1.5 B in and 2 B
// out per weight.
#pragma once

#include "w12_device.cuh"
#include "w12_format.hpp"

namespace w12 {
namespace dev {

struct DecodeParams {
    const uint8_t *blob;
    uint64_t off_seg, off_w, off_esc;
    int64_t N, K, chunks, segs;
    uint16_t *out;  // N x K row-major
};

__global__ void __launch_bounds__(128) w12_decode_kernel(const __grid_constant__ DecodeParams p) {
    // 128 rows x 64 bytes; 16-byte piece g of row r sits at piece
    // g ^ ((r >> 1) & 3), so both the row-wise writes of eight consecutive
    // lanes and the 2-rows-by-4-pieces reads of eight lanes hit distinct banks
    __shared__ __align__(16) uint8_t stage[kTileRows * 64];
    const int seg = blockIdx.x;
    const int64_t tile = blockIdx.y;
    const int q = threadIdx.x >> 5;
    const int r = threadIdx.x;

    const uint8_t *hp = p.blob + p.off_seg + (uint64_t)(tile * p.segs + seg) * kSegHdrBytes;
    const uint4 traw = __ldg(reinterpret_cast<const uint4 *>(hp));
    const uint4 meta = __ldg(reinterpret_cast<const uint4 *>(hp + 16));
    const Table T = make_table(traw);
    const uint32_t base = meta.x;
    const uint32_t qc0 = meta.y & 0xFFFFu, qc1 = meta.y >> 16, qc2 = meta.z & 0xFFFFu;
    const uint32_t mask = (meta.w >> (8 * q)) & 0xFFu;
    uint32_t run = base + (q > 0 ? qc0 : 0u) + (q > 1 ? qc1 : 0u) + (q > 2 ? qc2 : 0u);
    const uint8_t *esc = p.blob + p.off_esc;

    const int64_t n = tile * kTileRows + r;
    const int64_t left = p.chunks - (int64_t)seg * kChunksPerSeg;
    const int nch = (int)(left < kChunksPerSeg ? left : kChunksPerSeg);
    const bool vec_ok = ((p.K & 7) == 0) && ((reinterpret_cast<uintptr_t>(p.out) & 15) == 0);

    for (int j = 0; j < nch; ++j) {
        const int64_t chunk = (int64_t)seg * kChunksPerSeg + j;
        const uint8_t *cp = p.blob + p.off_w + (uint64_t)(tile * p.chunks + chunk) * kChunkBytes;
        const uint4 s_lo = __ldg(reinterpret_cast<const uint4 *>(cp + 16 * r));
        const uint4 s_hi = __ldg(reinterpret_cast<const uint4 *>(cp + kSlabBytes + 16 * r));
        const uint4 codes = __ldg(reinterpret_cast<const uint4 *>(cp + 2 * kSlabBytes + 16 * r));
        uint32_t E[8];
        decode_exponents(T, codes, E);
        if ((mask >> j) & 1u) run += warp_escapes(codes, esc + run, E);
        uint32_t out[16];
        assemble(s_lo, s_hi, E, out);

        const int64_t k0 = chunk * kChunkK;
        if (vec_ok && k0 + kChunkK <= p.K) {
            // stage this warp's 32 rows, then write them 8 rows x 64 bytes at a
            // time: lane l takes row 8i + l / 4 of the quarter, bytes 16 (l % 4)
            const int lane = r & 31;
#pragma unroll
            for (int g = 0; g < 4; ++g)
                *reinterpret_cast<uint4 *>(stage + 64 * r + 16 * (g ^ ((r >> 1) & 3))) =
                    make_uint4(out[4 * g], out[4 * g + 1], out[4 * g + 2], out[4 * g + 3]);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int rr = 32 * q + 8 * i + (lane >> 2);
                const int64_t nn = tile * kTileRows + rr;
                const uint4 v = *reinterpret_cast<const uint4 *>(stage + 64 * rr + 16 * ((lane & 3) ^ ((rr >> 1) & 3)));
                if (nn < p.N) *reinterpret_cast<uint4 *>(p.out + nn * p.K + k0 + 8 * (lane & 3)) = v;
            }
            __syncwarp();  // the stage is rewritten by the next chunk
        } else if (n < p.N) {
            uint16_t *dst = p.out + n * p.K + k0;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (k0 + 2 * i < p.K) dst[2 * i] = (uint16_t)(out[i] & 0xFFFFu);
                if (k0 + 2 * i + 1 < p.K) dst[2 * i + 1] = (uint16_t)(out[i] >> 16);
            }
        }
    }
}

}  // namespace dev
}  // namespace w12
