// Host side of the Q8 weight copy (format and scheme in include/w12.h): the
// quantizer and the header parser.  Rows are independent; a pool of host
// threads takes 128-row tiles.  Every float operation is plain IEEE fp32
// (division, rint to nearest even), so any conforming encoder writes the
// same bytes.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

#include "w12_host.hpp"

namespace w12 {
namespace host {
namespace {

inline void put_le(uint8_t *p, uint64_t v, int n) {
    for (int i = 0; i < n; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
inline uint64_t get_le(const uint8_t *p, int n) {
    uint64_t v = 0;
    for (int i = 0; i < n; ++i) v |= (uint64_t)p[i] << (8 * i);
    return v;
}
inline float bf16_to_float(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

// Quantizes tile t (rows 128t .. 128t+127); false if a row is not finite.
bool quantize_tile(const uint16_t *w, const q8::Geometry &g, int64_t t, uint8_t *blob) {
    for (int r = 0; r < kTileRows; ++r) {
        const int64_t n = t * kTileRows + r;
        if (n >= g.N) break;  // pad rows stay 0 (scale 0, q 0)
        const uint16_t *row = w + n * g.K;
        float a = 0.0f;
        for (int64_t k = 0; k < g.K; ++k) {
            const float v = bf16_to_float(row[k]);
            if (!std::isfinite(v)) return false;
            a = std::max(a, std::fabs(v));
        }
        const float s = a / 127.0f;
        std::memcpy(blob + g.off_s + 4 * (uint64_t)n, &s, 4);
        if (a == 0.0f) continue;  // q stays 0
        for (int64_t k = 0; k < g.K; ++k) {
            float q = std::rint(bf16_to_float(row[k]) / s);
            q = std::min(127.0f, std::max(-127.0f, q));
            const int64_t c = k / kChunkK, col = k % kChunkK;
            blob[g.off_q + (uint64_t)q8::kChunkBytes * (uint64_t)(t * g.chunks + c) +
                 (uint64_t)(kSlabBytes * (col / 16) + 16 * r + col % 16)] = (uint8_t)(int8_t)(int)q;
        }
    }
    return true;
}

}  // namespace

int q8_encoded_size(int64_t N, int64_t K, uint64_t *bytes, std::string *err) {
    if (!check_shape(N, K, err)) return W12_ERR_SHAPE;
    *bytes = q8::Geometry::of(N, K).total;
    return W12_OK;
}

int q8_encode(const uint16_t *w, int64_t N, int64_t K, uint8_t *blob, uint64_t cap, std::string *err) {
    if (!w || !blob) {
        *err = "null pointer";
        return W12_ERR_INVALID_ARG;
    }
    if (!check_shape(N, K, err)) return W12_ERR_SHAPE;
    const q8::Geometry g = q8::Geometry::of(N, K);
    if (cap < g.total) {
        *err = "blob buffer smaller than the Q8 size";
        return W12_ERR_BUFFER_TOO_SMALL;
    }
    std::memset(blob, 0, g.total);
    std::atomic<int64_t> next{0};
    std::atomic<bool> finite{true};
    const unsigned hw = std::thread::hardware_concurrency();
    const int64_t workers = std::min<int64_t>(g.tiles, hw ? std::min(hw, 128u) : 1u);
    auto work = [&] {
        for (int64_t t = next++; t < g.tiles; t = next++)
            if (!quantize_tile(w, g, t, blob)) finite = false;
    };
    if (workers <= 1) {
        work();
    } else {
        std::vector<std::thread> pool;
        for (int64_t i = 0; i < workers; ++i) pool.emplace_back(work);
        for (auto &th : pool) th.join();
    }
    if (!finite) {
        *err = "a weight is Inf or NaN: the row cannot be quantized";
        return W12_ERR_INVALID_ARG;
    }
    put_le(blob + q8::hdr::kMagicOff, q8::kMagic, 4);
    put_le(blob + q8::hdr::kVersionOff, q8::kVersion, 4);
    put_le(blob + q8::hdr::kHeaderBytesOff, kHeaderBytes, 4);
    put_le(blob + q8::hdr::kN, (uint64_t)g.N, 8);
    put_le(blob + q8::hdr::kK, (uint64_t)g.K, 8);
    put_le(blob + q8::hdr::kNpad, (uint64_t)g.Npad, 8);
    put_le(blob + q8::hdr::kKpad, (uint64_t)g.Kpad, 8);
    put_le(blob + q8::hdr::kTiles, (uint64_t)g.tiles, 8);
    put_le(blob + q8::hdr::kChunks, (uint64_t)g.chunks, 8);
    put_le(blob + q8::hdr::kOffS, g.off_s, 8);
    put_le(blob + q8::hdr::kBytesS, g.bytes_s, 8);
    put_le(blob + q8::hdr::kOffQ, g.off_q, 8);
    put_le(blob + q8::hdr::kBytesQ, g.bytes_q, 8);
    put_le(blob + q8::hdr::kTotal, g.total, 8);
    return W12_OK;
}

int q8_parse_header(const uint8_t *blob, uint64_t bytes, w12_q8_info *out, std::string *err) {
    if (!blob || !out) {
        *err = "null pointer";
        return W12_ERR_INVALID_ARG;
    }
    if (bytes < (uint64_t)kHeaderBytes) {
        *err = "blob shorter than its 256-byte header";
        return W12_ERR_BUFFER_TOO_SMALL;
    }
    if (get_le(blob + q8::hdr::kMagicOff, 4) != q8::kMagic || get_le(blob + q8::hdr::kVersionOff, 4) != q8::kVersion ||
        get_le(blob + q8::hdr::kHeaderBytesOff, 4) != (uint64_t)kHeaderBytes) {
        *err = "not a Q8 v1 blob (magic, version or header size)";
        return W12_ERR_CORRUPT_BLOB;
    }
    const int64_t N = (int64_t)get_le(blob + q8::hdr::kN, 8), K = (int64_t)get_le(blob + q8::hdr::kK, 8);
    if (!check_shape(N, K, err)) return W12_ERR_CORRUPT_BLOB;
    const q8::Geometry g = q8::Geometry::of(N, K);
    const bool ok = get_le(blob + q8::hdr::kFlagsOff, 4) == 0 &&
                    (int64_t)get_le(blob + q8::hdr::kNpad, 8) == g.Npad &&
                    (int64_t)get_le(blob + q8::hdr::kKpad, 8) == g.Kpad &&
                    (int64_t)get_le(blob + q8::hdr::kTiles, 8) == g.tiles &&
                    (int64_t)get_le(blob + q8::hdr::kChunks, 8) == g.chunks &&
                    get_le(blob + q8::hdr::kOffS, 8) == g.off_s && get_le(blob + q8::hdr::kBytesS, 8) == g.bytes_s &&
                    get_le(blob + q8::hdr::kOffQ, 8) == g.off_q && get_le(blob + q8::hdr::kBytesQ, 8) == g.bytes_q &&
                    get_le(blob + q8::hdr::kTotal, 8) == g.total;
    if (!ok) {
        *err = "Q8 header fields disagree with the geometry implied by N and K";
        return W12_ERR_CORRUPT_BLOB;
    }
    if (bytes < g.total) {
        *err = "blob buffer shorter than the blob's total size";
        return W12_ERR_BUFFER_TOO_SMALL;
    }
    out->N = g.N;
    out->K = g.K;
    out->N_pad = g.Npad;
    out->K_pad = g.Kpad;
    out->tiles = g.tiles;
    out->chunks = g.chunks;
    out->segs = g.segs;
    out->off_scales = g.off_s;
    out->bytes_scales = g.bytes_s;
    out->off_q = g.off_q;
    out->bytes_q = g.bytes_q;
    out->total_bytes = g.total;
    return W12_OK;
}

}  // namespace host
}  // namespace w12
