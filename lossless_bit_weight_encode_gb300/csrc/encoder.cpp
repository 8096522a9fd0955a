// Host encoder and blob checks of the W12 library (W12 v1, see include/w12.h).
//
// The encoder works one segment (128 rows x 256 columns) at a time, in two
// passes over all segments on every host core:
//   pass 1  exponent histogram -> table -> exponent-to-code map, escape count
//           per quarter and per chunk;
//   (prefix sum of the escape counts gives each segment's first escape slot)
//   pass 2  S bytes, 4-bit codes and escape bytes written in the escape order
//           (quarter, chunk, row, column), which also visits every packed row
//           exactly once.
// The output is canonical (same bytes as any other W12 v1 encoder).
// Properties the format must have: lossless and bit-exact ("StargazerX0/
// SpecPilot" §What it is, "SpecPilot" §Differentiation), ~12 bits per weight
// ("SpecPilot: an agent doubled speculative decoding speed, and the 10.87x
// needs context" §The mechanisms it found).
#include "w12_host.hpp"

#include <algorithm>
#include <atomic>
#include <cstring>
#include <thread>
#include <vector>

namespace w12 {
namespace host {
namespace {

struct SegPlan {
    uint8_t table[16];
    uint8_t code_of[256];
    uint16_t qcount[4];
    uint32_t chunk_mask;
};

inline void put_le(uint8_t *p, uint64_t v, int n) {
    for (int i = 0; i < n; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
inline uint64_t get_le(const uint8_t *p, int n) {
    uint64_t v = 0;
    for (int i = 0; i < n; ++i) v |= (uint64_t)p[i] << (8 * i);
    return v;
}

// Runs fn(i) for i in [0, n) on all host cores.
template <class Fn>
void parallel_for(int64_t n, Fn fn) {
    unsigned hw = std::thread::hardware_concurrency();
    int64_t workers = std::min<int64_t>(n, hw ? std::min(hw, 128u) : 1u);
    if (workers <= 1) {
        for (int64_t i = 0; i < n; ++i) fn(i);
        return;
    }
    std::atomic<int64_t> next{0};
    std::vector<std::thread> pool;
    pool.reserve((size_t)workers);
    for (int64_t t = 0; t < workers; ++t)
        pool.emplace_back([&] {
            for (int64_t i = next++; i < n; i = next++) fn(i);
        });
    for (auto &th : pool) th.join();
}

// Exponent histogram of segment (tile, seg), padded weights (+0.0) included.
void histogram(const uint16_t *w, const Geometry &g, int64_t tile, int64_t seg,
               uint32_t hist[256]) {
    std::memset(hist, 0, 256 * sizeof(uint32_t));
    const int64_t k0 = seg * kSegK;
    const int64_t k1 = std::min<int64_t>(k0 + kSegK, g.Kpad);
    const int64_t kreal = std::max<int64_t>(0, std::min<int64_t>(k1, g.K) - k0);
    uint64_t pads = 0;
    for (int r = 0; r < kTileRows; ++r) {
        const int64_t n = tile * kTileRows + r;
        if (n >= g.N) {
            pads += (uint64_t)(k1 - k0);
            continue;
        }
        const uint16_t *row = w + n * g.K + k0;
        for (int64_t k = 0; k < kreal; ++k) hist[(row[k] >> 7) & 0xFF]++;
        pads += (uint64_t)(k1 - k0 - kreal);
    }
    hist[0] += (uint32_t)pads;
}

// Table of a segment from its histogram (the format's ranking and slot rule).
void make_table(const uint32_t hist[256], uint8_t table[16]) {
    // key: count in the high bits, then 255 - exponent so that the smaller
    // exponent wins a tie when sorting by key, largest first
    uint64_t keys[256];
    int nkeys = 0;
    for (int e = 0; e < 256; ++e)
        if (hist[e]) keys[nkeys++] = ((uint64_t)hist[e] << 8) | (uint64_t)(255 - e);
    const int take = std::min(nkeys, 15);
    std::partial_sort(keys, keys + take, keys + nkeys, [](uint64_t a, uint64_t b) { return a > b; });
    bool chosen[256] = {};
    for (int i = 0; i < take; ++i) chosen[255 - (int)(keys[i] & 0xFF)] = true;

    uint8_t low[15], high[15];
    int nlow = 0, nhigh = 0;
    for (int e = 0; e < 256; ++e) {
        if (!chosen[e]) continue;
        if (e & 0x80) high[nhigh++] = (uint8_t)e;
        else low[nlow++] = (uint8_t)e;
    }
    // Slot 7 is paired with the escape slot; slots j and j + 8 form pairs.
    static constexpr int kVisit[15] = {7, 0, 8, 1, 9, 2, 10, 3, 11, 4, 12, 5, 13, 6, 14};
    const bool low_first = (nlow & 1) || !(nhigh & 1);
    const int start = ((nlow & 1) || (nhigh & 1)) ? 0 : 1;
    int16_t slot[16];
    for (int i = 0; i < 16; ++i) slot[i] = -1;
    int pos = start;
    auto place = [&](const uint8_t *v, int n) {
        for (int i = 0; i < n; ++i) slot[kVisit[pos++]] = v[i];
    };
    if (low_first) {
        place(low, nlow);
        place(high, nhigh);
    } else {
        place(high, nhigh);
        place(low, nlow);
    }
    for (int c = 0; c < 15; ++c) {
        if (slot[c] >= 0) {
            table[c] = (uint8_t)slot[c];
            continue;
        }
        const int partner = (c == 7) ? 15 : (c ^ 8);
        table[c] = slot[partner] >= 0 ? (uint8_t)slot[partner] : 0;
    }
    table[15] = 0;
}

// Pass 1 for one segment: table, code map, escape counts and chunk mask.
void plan_segment(const uint16_t *w, const Geometry &g, int64_t tile, int64_t seg, SegPlan &p) {
    uint32_t hist[256];
    histogram(w, g, tile, seg, hist);
    make_table(hist, p.table);
    std::memset(p.code_of, 15, sizeof p.code_of);
    for (int c = 14; c >= 0; --c) p.code_of[p.table[c]] = (uint8_t)c;  // first slot wins
    p.chunk_mask = 0;
    const int nch = g.seg_chunks(seg);
    for (int q = 0; q < 4; ++q) {
        uint32_t cnt = 0;
        for (int j = 0; j < nch; ++j) {
            const int64_t k0 = (seg * kChunksPerSeg + j) * (int64_t)kChunkK;
            uint32_t cj = 0;
            for (int r = q * kQuarterRows; r < (q + 1) * kQuarterRows; ++r) {
                const int64_t n = tile * kTileRows + r;
                for (int kk = 0; kk < kChunkK; ++kk) {
                    const int64_t k = k0 + kk;
                    const uint16_t b = (n < g.N && k < g.K) ? w[n * g.K + k] : 0;
                    cj += p.code_of[(b >> 7) & 0xFF] == 15;
                }
            }
            if (cj) p.chunk_mask |= 1u << (8 * q + j);
            cnt += cj;
        }
        p.qcount[q] = (uint16_t)cnt;
    }
}

// Pass 2 for one segment: its header, packed rows and escape bytes.
void write_segment(const uint16_t *w, const Geometry &g, int64_t tile, int64_t seg,
                   const SegPlan &p, uint32_t esc_base, uint8_t *blob) {
    SegHeader h;
    std::memcpy(h.table, p.table, 16);
    h.esc_base = esc_base;
    for (int q = 0; q < 4; ++q) h.qcount[q] = p.qcount[q];
    h.chunk_mask = p.chunk_mask;
    uint8_t *hp = blob + g.off_seg + (uint64_t)(tile * g.segs + seg) * kSegHdrBytes;
    std::memcpy(hp, h.table, 16);
    put_le(hp + 16, h.esc_base, 4);
    for (int q = 0; q < 4; ++q) put_le(hp + 20 + 2 * q, h.qcount[q], 2);
    put_le(hp + 28, h.chunk_mask, 4);

    uint8_t *esc = blob + g.off_esc + esc_base;
    const int nch = g.seg_chunks(seg);
    uint16_t v[kChunkK];
    for (int q = 0; q < 4; ++q) {
        for (int j = 0; j < nch; ++j) {
            const int64_t chunk = seg * kChunksPerSeg + j;
            const int64_t k0 = chunk * kChunkK;
            uint8_t *cp = blob + g.off_w + (uint64_t)(tile * g.chunks + chunk) * kChunkBytes;
            for (int r = q * kQuarterRows; r < (q + 1) * kQuarterRows; ++r) {
                const int64_t n = tile * kTileRows + r;
                if (n < g.N && k0 + kChunkK <= g.K) {
                    std::memcpy(v, w + n * g.K + k0, sizeof v);
                } else {
                    for (int kk = 0; kk < kChunkK; ++kk)
                        v[kk] = (n < g.N && k0 + kk < g.K) ? w[n * g.K + k0 + kk] : 0;
                }
                uint8_t *s_lo = cp + 16 * r;
                uint8_t *s_hi = cp + kSlabBytes + 16 * r;
                uint8_t *codes = cp + 2 * kSlabBytes + 16 * r;
                for (int kk = 0; kk < kChunkK; kk += 2) {
                    const uint16_t a = v[kk], b = v[kk + 1];
                    const uint8_t sa = (uint8_t)(((a & 0x7F) << 1) | (b >> 15));
                    const uint8_t sb = (uint8_t)(((b & 0x7F) << 1) | (a >> 15));
                    uint8_t *sdst = kk < 16 ? s_lo + kk : s_hi + (kk - 16);
                    sdst[0] = sa;
                    sdst[1] = sb;
                    const uint8_t ea = (uint8_t)(a >> 7), eb = (uint8_t)(b >> 7);
                    const uint8_t ca = p.code_of[ea], cb = p.code_of[eb];
                    codes[kk >> 1] = (uint8_t)(ca | (cb << 4));
                    if (ca == 15) *esc++ = ea;
                    if (cb == 15) *esc++ = eb;
                }
            }
        }
    }
}

}  // namespace

bool check_shape(int64_t N, int64_t K, std::string *err) {
    // Keeps every offset well inside 63 bits and N*K representable.
    if (N < 1 || K < 1 || N > (int64_t(1) << 31) || K > (int64_t(1) << 31) ||
        (N / 128 + 1) * (K / 32 + 1) > (int64_t(1) << 40)) {
        *err = "N and K must be in [1, 2^31] with a packed size below 2^52 bytes";
        return false;
    }
    return true;
}

int encoded_size(const uint16_t *w, int64_t N, int64_t K, uint64_t *bytes, std::string *err) {
    if (!w || !bytes) {
        *err = "null pointer";
        return W12_ERR_INVALID_ARG;
    }
    if (!check_shape(N, K, err)) return W12_ERR_SHAPE;
    const Geometry g = Geometry::of(N, K);
    const int64_t nseg = g.tiles * g.segs;
    std::vector<uint64_t> counts((size_t)nseg);
    parallel_for(nseg, [&](int64_t i) {
        SegPlan p;
        plan_segment(w, g, i / g.segs, i % g.segs, p);
        counts[(size_t)i] = (uint64_t)p.qcount[0] + p.qcount[1] + p.qcount[2] + p.qcount[3];
    });
    uint64_t total_esc = 0;
    for (uint64_t c : counts) total_esc += c;
    if (total_esc > 0xFFFFFFFFull) {
        *err = "more than 2^32-1 escapes: split the matrix";
        return W12_ERR_SHAPE;
    }
    *bytes = g.total(total_esc);
    return W12_OK;
}

int encode(const uint16_t *w, int64_t N, int64_t K, uint8_t *blob, uint64_t cap, std::string *err) {
    if (!w || !blob) {
        *err = "null pointer";
        return W12_ERR_INVALID_ARG;
    }
    if (!check_shape(N, K, err)) return W12_ERR_SHAPE;
    const Geometry g = Geometry::of(N, K);
    const int64_t nseg = g.tiles * g.segs;
    std::vector<SegPlan> plans((size_t)nseg);
    parallel_for(nseg, [&](int64_t i) { plan_segment(w, g, i / g.segs, i % g.segs, plans[(size_t)i]); });
    std::vector<uint64_t> base((size_t)nseg + 1, 0);
    for (int64_t i = 0; i < nseg; ++i) {
        const SegPlan &p = plans[(size_t)i];
        base[(size_t)i + 1] = base[(size_t)i] + p.qcount[0] + p.qcount[1] + p.qcount[2] + p.qcount[3];
    }
    const uint64_t n_esc = base[(size_t)nseg];
    if (n_esc > 0xFFFFFFFFull) {
        *err = "more than 2^32-1 escapes: split the matrix";
        return W12_ERR_SHAPE;
    }
    const uint64_t total = g.total(n_esc);
    if (cap < total) {
        *err = "blob buffer smaller than the encoded size";
        return W12_ERR_BUFFER_TOO_SMALL;
    }
    // zero the header and all alignment gaps; the planes are written in full
    std::memset(blob, 0, g.off_w);
    std::memset(blob + g.off_w + g.bytes_w, 0, g.off_esc - (g.off_w + g.bytes_w));
    std::memset(blob + g.off_esc + n_esc, 0, total - (g.off_esc + n_esc));
    parallel_for(nseg, [&](int64_t i) {
        write_segment(w, g, i / g.segs, i % g.segs, plans[(size_t)i], (uint32_t)base[(size_t)i], blob);
    });

    put_le(blob + hdr::kMagicOff, kMagic, 4);
    put_le(blob + hdr::kVersionOff, kVersion, 4);
    put_le(blob + hdr::kHeaderBytesOff, kHeaderBytes, 4);
    put_le(blob + hdr::kN, (uint64_t)g.N, 8);
    put_le(blob + hdr::kK, (uint64_t)g.K, 8);
    put_le(blob + hdr::kNpad, (uint64_t)g.Npad, 8);
    put_le(blob + hdr::kKpad, (uint64_t)g.Kpad, 8);
    put_le(blob + hdr::kTileRowsOff, kTileRows, 4);
    put_le(blob + hdr::kChunkKOff, kChunkK, 4);
    put_le(blob + hdr::kSegKOff, kSegK, 4);
    put_le(blob + hdr::kQuarterOff, kQuarterRows, 4);
    put_le(blob + hdr::kTiles, (uint64_t)g.tiles, 8);
    put_le(blob + hdr::kChunks, (uint64_t)g.chunks, 8);
    put_le(blob + hdr::kSegs, (uint64_t)g.segs, 8);
    put_le(blob + hdr::kOffSeg, g.off_seg, 8);
    put_le(blob + hdr::kBytesSeg, g.bytes_seg, 8);
    put_le(blob + hdr::kOffW, g.off_w, 8);
    put_le(blob + hdr::kBytesW, g.bytes_w, 8);
    put_le(blob + hdr::kOffEsc, g.off_esc, 8);
    put_le(blob + hdr::kNEsc, n_esc, 8);
    put_le(blob + hdr::kBytesEsc, g.bytes_esc(n_esc), 8);
    put_le(blob + hdr::kTotal, total, 8);
    return W12_OK;
}

int parse_header(const uint8_t *blob, uint64_t bytes, w12_info *out, std::string *err) {
    if (!blob || !out) {
        *err = "null pointer";
        return W12_ERR_INVALID_ARG;
    }
    if (bytes < (uint64_t)kHeaderBytes) {
        *err = "blob shorter than its 256-byte header";
        return W12_ERR_BUFFER_TOO_SMALL;
    }
    if (get_le(blob + hdr::kMagicOff, 4) != kMagic) {
        *err = "bad magic (not a W12 blob)";
        return W12_ERR_CORRUPT_BLOB;
    }
    if (get_le(blob + hdr::kVersionOff, 4) != kVersion || get_le(blob + hdr::kHeaderBytesOff, 4) != (uint64_t)kHeaderBytes) {
        *err = "unsupported W12 version or header size";
        return W12_ERR_CORRUPT_BLOB;
    }
    const int64_t N = (int64_t)get_le(blob + hdr::kN, 8), K = (int64_t)get_le(blob + hdr::kK, 8);
    if (!check_shape(N, K, err)) return W12_ERR_CORRUPT_BLOB;
    const Geometry g = Geometry::of(N, K);
    const uint64_t n_esc = get_le(blob + hdr::kNEsc, 8);
    const bool ok =
        get_le(blob + hdr::kFlagsOff, 4) == 0 &&
        (int64_t)get_le(blob + hdr::kNpad, 8) == g.Npad && (int64_t)get_le(blob + hdr::kKpad, 8) == g.Kpad &&
        get_le(blob + hdr::kTileRowsOff, 4) == (uint64_t)kTileRows &&
        get_le(blob + hdr::kChunkKOff, 4) == (uint64_t)kChunkK &&
        get_le(blob + hdr::kSegKOff, 4) == (uint64_t)kSegK &&
        get_le(blob + hdr::kQuarterOff, 4) == (uint64_t)kQuarterRows &&
        (int64_t)get_le(blob + hdr::kTiles, 8) == g.tiles &&
        (int64_t)get_le(blob + hdr::kChunks, 8) == g.chunks &&
        (int64_t)get_le(blob + hdr::kSegs, 8) == g.segs &&
        get_le(blob + hdr::kOffSeg, 8) == g.off_seg && get_le(blob + hdr::kBytesSeg, 8) == g.bytes_seg &&
        get_le(blob + hdr::kOffW, 8) == g.off_w && get_le(blob + hdr::kBytesW, 8) == g.bytes_w &&
        get_le(blob + hdr::kOffEsc, 8) == g.off_esc && n_esc <= 0xFFFFFFFFull &&
        get_le(blob + hdr::kBytesEsc, 8) == g.bytes_esc(n_esc) &&
        get_le(blob + hdr::kTotal, 8) == g.total(n_esc);
    if (!ok) {
        *err = "header fields disagree with the geometry implied by N and K";
        return W12_ERR_CORRUPT_BLOB;
    }
    if (bytes < g.total(n_esc)) {
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
    out->off_seghdr = g.off_seg;
    out->bytes_seghdr = g.bytes_seg;
    out->off_weights = g.off_w;
    out->bytes_weights = g.bytes_w;
    out->off_escapes = g.off_esc;
    out->bytes_escapes = g.bytes_esc(n_esc);
    out->n_escapes = n_esc;
    out->total_bytes = g.total(n_esc);
    out->bits_per_weight = 8.0 * (double)out->total_bytes / ((double)N * (double)K);
    return W12_OK;
}

int validate(const uint8_t *blob, uint64_t bytes, std::string *err) {
    w12_info info;
    int rc = parse_header(blob, bytes, &info, err);
    if (rc != W12_OK) return rc;
    const Geometry g = Geometry::of(info.N, info.K);
    uint64_t running = 0;
    for (int64_t t = 0; t < g.tiles; ++t) {
        for (int64_t s = 0; s < g.segs; ++s) {
            const uint8_t *h = blob + g.off_seg + (uint64_t)(t * g.segs + s) * kSegHdrBytes;
            bool ok = h[15] == 0;
            for (int j = 0; j < 7; ++j) ok = ok && ((h[j] ^ h[j + 8]) & 0x80) == 0;
            ok = ok && get_le(h + 16, 4) == running;
            const uint32_t mask = (uint32_t)get_le(h + 28, 4);
            const int nch = g.seg_chunks(s);
            for (int q = 0; q < 4; ++q) {
                const uint32_t qc = (uint32_t)get_le(h + 20 + 2 * q, 2);
                const uint32_t qmask = (mask >> (8 * q)) & 0xFFu;
                ok = ok && (qc == 0) == (qmask == 0);
                ok = ok && (qmask >> nch) == 0;
                ok = ok && qc <= (uint32_t)(kQuarterRows * kChunkK * nch);
                ok = ok && (uint32_t)__builtin_popcount(qmask) <= qc;
                running += qc;
            }
            if (!ok) {
                *err = "segment header " + std::to_string(t) + "," + std::to_string(s) + " is inconsistent";
                return W12_ERR_CORRUPT_BLOB;
            }
        }
    }
    if (running != info.n_escapes) {
        *err = "segment escape counts do not add up to the header's escape count";
        return W12_ERR_CORRUPT_BLOB;
    }
    return W12_OK;
}

}  // namespace host
}  // namespace w12
