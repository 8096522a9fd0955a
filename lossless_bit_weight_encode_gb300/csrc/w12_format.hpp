// W12 v1 format constants and blob geometry shared by the host encoder, the
// C ABI and the kernels of the library.  (The test oracle keeps its own copy.)
//
// Format definition: see include/w12.h.  Sources for the properties the format
// must have: "StargazerX0/SpecPilot" (hotrepo.ai) §What it is; "SpecPilot"
// (fasttoolhub.com) §Differentiation; "SpecPilot: an agent doubled speculative
// decoding speed, and the 10.87x needs context" (ai.jakubjirak.com) §The
// mechanisms it found.
#pragma once

#include <cstdint>

namespace w12 {

constexpr int kTileRows = 128;
constexpr int kQuarterRows = 32;
constexpr int kChunkK = 32;
constexpr int kSegK = 256;
constexpr int kChunksPerSeg = kSegK / kChunkK;   // 8
constexpr int kSlabBytes = kTileRows * 16;       // 2048
constexpr int kChunkBytes = 3 * kSlabBytes;      // 6144
constexpr int kSegHdrBytes = 32;
constexpr int kHeaderBytes = 256;
constexpr int kPlaneAlign = 256;
constexpr uint32_t kMagic = 0x42323157u;         // "W12B" little-endian
constexpr uint32_t kVersion = 1;

// Header field offsets.
namespace hdr {
constexpr int kMagicOff = 0x00, kVersionOff = 0x04, kHeaderBytesOff = 0x08, kFlagsOff = 0x0C;
constexpr int kN = 0x10, kK = 0x18, kNpad = 0x20, kKpad = 0x28;
constexpr int kTileRowsOff = 0x30, kChunkKOff = 0x34, kSegKOff = 0x38, kQuarterOff = 0x3C;
constexpr int kTiles = 0x40, kChunks = 0x48, kSegs = 0x50;
constexpr int kOffSeg = 0x58, kBytesSeg = 0x60, kOffW = 0x68, kBytesW = 0x70;
constexpr int kOffEsc = 0x78, kNEsc = 0x80, kBytesEsc = 0x88, kTotal = 0x90;
}  // namespace hdr

// Segment header layout (32 bytes).
struct SegHeader {
    uint8_t table[16];
    uint32_t esc_base;
    uint16_t qcount[4];
    uint32_t chunk_mask;
};
static_assert(sizeof(SegHeader) == kSegHdrBytes, "segment header is 32 bytes");

struct Geometry {
    int64_t N = 0, K = 0, Npad = 0, Kpad = 0;
    int64_t tiles = 0, chunks = 0, segs = 0;
    uint64_t off_seg = 0, bytes_seg = 0, off_w = 0, bytes_w = 0, off_esc = 0;

    static inline uint64_t round_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

    // Fills every plane offset that does not depend on the escape count.
    static inline Geometry of(int64_t n, int64_t k) {
        Geometry g;
        g.N = n;
        g.K = k;
        g.Npad = (int64_t)round_up((uint64_t)n, kTileRows);
        g.Kpad = (int64_t)round_up((uint64_t)k, kChunkK);
        g.tiles = g.Npad / kTileRows;
        g.chunks = g.Kpad / kChunkK;
        g.segs = (g.chunks + kChunksPerSeg - 1) / kChunksPerSeg;
        g.off_seg = kHeaderBytes;
        g.bytes_seg = (uint64_t)kSegHdrBytes * (uint64_t)(g.tiles * g.segs);
        g.off_w = round_up(g.off_seg + g.bytes_seg, kPlaneAlign);
        g.bytes_w = (uint64_t)kChunkBytes * (uint64_t)(g.tiles * g.chunks);
        g.off_esc = round_up(g.off_w + g.bytes_w, kPlaneAlign);
        return g;
    }
    inline uint64_t bytes_esc(uint64_t n_esc) const { return round_up(n_esc, 16); }
    inline uint64_t total(uint64_t n_esc) const {
        return round_up(off_esc + bytes_esc(n_esc), kPlaneAlign);
    }
    // Chunks in segment s of any tile (the last segment may be short).
    inline int seg_chunks(int64_t s) const {
        int64_t left = chunks - s * kChunksPerSeg;
        return (int)(left < kChunksPerSeg ? left : kChunksPerSeg);
    }
};

// Q8 v1: the 8-bit weight copy (symmetric INT8 per row, fp32 scale per row;
// format in include/w12.h).  Same tile/chunk/segment grid as W12; a chunk is
// two slabs of 128 rows x 16 int8 (columns 0-15, 16-31).
namespace q8 {
constexpr int kChunkBytes = 2 * kSlabBytes;      // 4096
constexpr uint32_t kMagic = 0x31573851u;         // "Q8W1" little-endian
constexpr uint32_t kVersion = 1;
namespace hdr {
constexpr int kMagicOff = 0x00, kVersionOff = 0x04, kHeaderBytesOff = 0x08, kFlagsOff = 0x0C;
constexpr int kN = 0x10, kK = 0x18, kNpad = 0x20, kKpad = 0x28, kTiles = 0x30, kChunks = 0x38;
constexpr int kOffS = 0x40, kBytesS = 0x48, kOffQ = 0x50, kBytesQ = 0x58, kTotal = 0x60;
}  // namespace hdr

struct Geometry {
    int64_t N = 0, K = 0, Npad = 0, Kpad = 0, tiles = 0, chunks = 0, segs = 0;
    uint64_t off_s = 0, bytes_s = 0, off_q = 0, bytes_q = 0, total = 0;

    static inline Geometry of(int64_t n, int64_t k) {
        Geometry g;
        g.N = n;
        g.K = k;
        g.Npad = (int64_t)w12::Geometry::round_up((uint64_t)n, kTileRows);
        g.Kpad = (int64_t)w12::Geometry::round_up((uint64_t)k, kChunkK);
        g.tiles = g.Npad / kTileRows;
        g.chunks = g.Kpad / kChunkK;
        g.segs = (g.chunks + kChunksPerSeg - 1) / kChunksPerSeg;
        g.off_s = kHeaderBytes;
        g.bytes_s = 4ull * (uint64_t)g.Npad;
        g.off_q = w12::Geometry::round_up(g.off_s + g.bytes_s, kPlaneAlign);
        g.bytes_q = (uint64_t)kChunkBytes * (uint64_t)(g.tiles * g.chunks);
        g.total = w12::Geometry::round_up(g.off_q + g.bytes_q, kPlaneAlign);
        return g;
    }
};
}  // namespace q8

}  // namespace w12
