// C ABI of the W12 library (declared in include/w12.h): argument checks,
// error strings, and dispatch to the host encoder and the kernel launchers.
// No exception crosses this boundary.
#include <cstdint>
#include <exception>
#include <string>

#include "w12.h"
#include "w12_host.hpp"
#include "w12_launch.hpp"

namespace {

thread_local std::string t_last_error;

int finish(int rc, const std::string &err) {
    t_last_error = rc == W12_OK ? std::string() : err;
    return rc;
}

template <class Fn>
int guarded(Fn fn) {
    try {
        std::string err;
        const int rc = fn(err);
        return finish(rc, err);
    } catch (const std::exception &e) {
        return finish(W12_ERR_INVALID_ARG, std::string("internal error: ") + e.what());
    } catch (...) {
        return finish(W12_ERR_INVALID_ARG, "internal error");
    }
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_info(const w12_info *info, std::string &err) {
    if (!info) {
        err = "info is null";
        return W12_ERR_INVALID_ARG;
    }
    if (info->N < 1 || info->K < 1 || info->tiles != info->N_pad / 128 || info->chunks != info->K_pad / 32 ||
        info->N_pad != (info->N + 127) / 128 * 128 || info->K_pad != (info->K + 31) / 32 * 32 ||
        info->segs != (info->chunks + 7) / 8) {
        err = "info does not describe a W12 v1 blob (fill it with w12_blob_info)";
        return W12_ERR_INVALID_ARG;
    }
    return W12_OK;
}

int check_q8_info(const w12_q8_info *info, std::string &err) {
    if (!info) {
        err = "info is null";
        return W12_ERR_INVALID_ARG;
    }
    const w12::q8::Geometry g = w12::q8::Geometry::of(info->N, info->K);
    if (info->N < 1 || info->K < 1 || info->tiles != g.tiles || info->chunks != g.chunks || info->segs != g.segs ||
        info->N_pad != g.Npad || info->K_pad != g.Kpad || info->off_scales != g.off_s || info->off_q != g.off_q ||
        info->total_bytes != g.total) {
        err = "info does not describe a Q8 v1 blob (fill it with w12_q8_blob_info)";
        return W12_ERR_INVALID_ARG;
    }
    return W12_OK;
}

}  // namespace

extern "C" {

const char *w12_last_error(void) { return t_last_error.c_str(); }

const char *w12_status_string(int status) {
    switch (status) {
    case W12_OK: return "W12_OK";
    case W12_ERR_INVALID_ARG: return "W12_ERR_INVALID_ARG";
    case W12_ERR_SHAPE: return "W12_ERR_SHAPE";
    case W12_ERR_BUFFER_TOO_SMALL: return "W12_ERR_BUFFER_TOO_SMALL";
    case W12_ERR_ALIGNMENT: return "W12_ERR_ALIGNMENT";
    case W12_ERR_CORRUPT_BLOB: return "W12_ERR_CORRUPT_BLOB";
    case W12_ERR_UNSUPPORTED_ARCH: return "W12_ERR_UNSUPPORTED_ARCH";
    case W12_ERR_CUDA: return "W12_ERR_CUDA";
    case W12_ERR_TIMEOUT: return "W12_ERR_TIMEOUT";
    default: return "W12_ERR_UNKNOWN";
    }
}

int w12_format_version(void) { return W12_FORMAT_VERSION; }

int w12_encoded_size_host(const uint16_t *w_host, int64_t N, int64_t K, size_t *bytes) {
    return guarded([&](std::string &err) {
        uint64_t b = 0;
        const int rc = w12::host::encoded_size(w_host, N, K, &b, &err);
        if (rc == W12_OK) *bytes = (size_t)b;
        return rc;
    });
}

int w12_encode_host(const uint16_t *w_host, int64_t N, int64_t K, void *blob_host, size_t bytes) {
    return guarded([&](std::string &err) {
        return w12::host::encode(w_host, N, K, static_cast<uint8_t *>(blob_host), bytes, &err);
    });
}

int w12_blob_info(const void *blob_host, size_t bytes, w12_info *out) {
    return guarded([&](std::string &err) {
        return w12::host::parse_header(static_cast<const uint8_t *>(blob_host), bytes, out, &err);
    });
}

int w12_blob_validate(const void *blob_host, size_t bytes) {
    return guarded([&](std::string &err) {
        return w12::host::validate(static_cast<const uint8_t *>(blob_host), bytes, &err);
    });
}

int w12_decode(const void *blob_dev, const w12_info *info, uint16_t *w_out_dev, void *stream) {
    return guarded([&](std::string &err) {
        int rc = check_info(info, err);
        if (rc != W12_OK) return rc;
        if (!blob_dev || !w_out_dev) {
            err = "null device pointer";
            return (int)W12_ERR_INVALID_ARG;
        }
        if (!aligned(blob_dev, 256) || !aligned(w_out_dev, 2)) {
            err = "blob_dev must be 256-byte aligned and w_out_dev 2-byte aligned";
            return (int)W12_ERR_ALIGNMENT;
        }
        return w12::launch::decode(blob_dev, *info, w_out_dev, stream, &err);
    });
}

int w12_gemm_workspace_size(const w12_info *info, int M, size_t *bytes) {
    return guarded([&](std::string &err) {
        int rc = check_info(info, err);
        if (rc != W12_OK) return rc;
        if (!bytes) {
            err = "bytes is null";
            return (int)W12_ERR_INVALID_ARG;
        }
        w12::launch::GemmPlan plan;
        rc = w12::launch::plan_gemm(*info, M, &plan, &err);
        if (rc == W12_OK) *bytes = plan.ws_bytes;
        return rc;
    });
}

int w12_gemm_launch_info(const w12_info *info, int M, int32_t out[4]) {
    return guarded([&](std::string &err) {
        int rc = check_info(info, err);
        if (rc != W12_OK) return rc;
        if (!out) {
            err = "out is null";
            return (int)W12_ERR_INVALID_ARG;
        }
        w12::launch::GemmPlan plan;
        rc = w12::launch::plan_gemm(*info, M, &plan, &err);
        if (rc == W12_OK) {
            out[0] = plan.ntok;
            out[1] = plan.splits;
            out[2] = plan.ctas;
            out[3] = plan.ctas_per_sm;
        }
        return rc;
    });
}

int w12_gemm(const uint16_t *x_dev, const void *blob_dev, const w12_info *info, uint16_t *y_dev, int M,
             void *workspace, size_t ws_bytes, void *stream) {
    return guarded([&](std::string &err) {
        int rc = check_info(info, err);
        if (rc != W12_OK) return rc;
        if (!x_dev || !blob_dev || !y_dev || !workspace) {
            err = "null device pointer";
            return (int)W12_ERR_INVALID_ARG;
        }
        if (M < 1 || M > 32) {
            err = "M must be in 1..32";
            return (int)W12_ERR_INVALID_ARG;
        }
        if (!aligned(blob_dev, 256) || !aligned(workspace, 256) || !aligned(y_dev, 2) || !aligned(x_dev, 2)) {
            err = "blob_dev and workspace must be 256-byte aligned, x_dev and y_dev 2-byte aligned";
            return (int)W12_ERR_ALIGNMENT;
        }
        return w12::launch::gemm(x_dev, blob_dev, *info, y_dev, M, workspace, ws_bytes, stream, &err);
    });
}

namespace {
int check_group(int count, const w12_info *infos, std::string &err) {
    if (count < 1 || count > W12_MAX_GROUP || !infos) {
        err = "count must be in 1.." + std::to_string(W12_MAX_GROUP) + " with non-null infos";
        return W12_ERR_INVALID_ARG;
    }
    for (int i = 0; i < count; ++i) {
        const int rc = check_info(&infos[i], err);
        if (rc != W12_OK) return rc;
        if (infos[i].K != infos[0].K) {
            err = "the matrices of a group must share K (they multiply the same x)";
            return W12_ERR_SHAPE;
        }
    }
    return W12_OK;
}
}  // namespace

int w12_gemm_group_launch_info(int count, const w12_info *infos, int M, int32_t out[5]) {
    return guarded([&](std::string &err) {
        int rc = check_group(count, infos, err);
        if (rc != W12_OK) return rc;
        if (!out) {
            err = "out is null";
            return (int)W12_ERR_INVALID_ARG;
        }
        w12::launch::GemmPlan plan;
        rc = w12::launch::group_plan(count, infos, M, &plan, &err);
        if (rc == W12_OK) {
            out[0] = plan.ntok;
            out[1] = plan.splits;
            out[2] = plan.ctas;
            out[3] = plan.ctas_per_sm;
            out[4] = plan.kernel;
        }
        return rc;
    });
}

int w12_gemm_group_workspace_size(int count, const w12_info *infos, int M, size_t *bytes) {
    return guarded([&](std::string &err) {
        int rc = check_group(count, infos, err);
        if (rc != W12_OK) return rc;
        if (!bytes || M < 1 || M > 32) {
            err = "null pointer or M outside 1..32";
            return (int)W12_ERR_INVALID_ARG;
        }
        return w12::launch::group_workspace_size(count, infos, M, bytes, &err);
    });
}

int w12_gemm_group(const uint16_t *x_dev, int count, const void *const *blobs_dev, const w12_info *infos,
                   uint16_t *const *y_devs, int M, void *workspace, size_t ws_bytes, void *stream) {
    return guarded([&](std::string &err) {
        int rc = check_group(count, infos, err);
        if (rc != W12_OK) return rc;
        if (!x_dev || !blobs_dev || !y_devs || !workspace) {
            err = "null pointer";
            return (int)W12_ERR_INVALID_ARG;
        }
        if (M < 1 || M > 32) {
            err = "M must be in 1..32";
            return (int)W12_ERR_INVALID_ARG;
        }
        if (!aligned(workspace, 256) || !aligned(x_dev, 2)) {
            err = "workspace must be 256-byte aligned and x_dev 2-byte aligned";
            return (int)W12_ERR_ALIGNMENT;
        }
        for (int i = 0; i < count; ++i) {
            if (!blobs_dev[i] || !y_devs[i]) {
                err = "null blob or output";
                return (int)W12_ERR_INVALID_ARG;
            }
            if (!aligned(blobs_dev[i], 256) || !aligned(y_devs[i], 2)) {
                err = "each blob must be 256-byte aligned and each y 2-byte aligned";
                return (int)W12_ERR_ALIGNMENT;
            }
        }
        return w12::launch::gemm_group(x_dev, count, blobs_dev, infos, y_devs, M, workspace, ws_bytes, stream, &err);
    });
}

int w12_gemm_argmax_workspace_size(const w12_info *info, int M, size_t *bytes) {
    return guarded([&](std::string &err) {
        int rc = check_info(info, err);
        if (rc != W12_OK) return rc;
        if (!bytes || M < 1 || M > 32) {
            err = "null pointer or M outside 1..32";
            return (int)W12_ERR_INVALID_ARG;
        }
        return w12::launch::argmax_workspace_size(*info, M, bytes, &err);
    });
}

int w12_gemm_argmax(const uint16_t *x_dev, const void *blob_dev, const w12_info *info, int M, uint16_t *y_dev,
                    int32_t *idx_dev, float *val_dev, void *workspace, size_t ws_bytes, void *stream) {
    return guarded([&](std::string &err) {
        int rc = check_info(info, err);
        if (rc != W12_OK) return rc;
        if (!x_dev || !blob_dev || !idx_dev || !val_dev || !workspace) {
            err = "null device pointer";
            return (int)W12_ERR_INVALID_ARG;
        }
        if (M < 1 || M > 32) {
            err = "M must be in 1..32";
            return (int)W12_ERR_INVALID_ARG;
        }
        if (info->N > 0x7FFFFFFF) {
            err = "N must fit in int32 for the argmax index";
            return (int)W12_ERR_SHAPE;
        }
        if (!aligned(blob_dev, 256) || !aligned(workspace, 256) || !aligned(x_dev, 2) || !aligned(y_dev, 2) ||
            !aligned(idx_dev, 4) || !aligned(val_dev, 4)) {
            err = "blob_dev and workspace must be 256-byte aligned, x_dev and y_dev 2-byte, idx and val 4-byte";
            return (int)W12_ERR_ALIGNMENT;
        }
        return w12::launch::gemm_argmax(x_dev, blob_dev, *info, M, y_dev, idx_dev, val_dev, workspace, ws_bytes,
                                        stream, &err);
    });
}

int w12_gemm_noalloc(const uint16_t *x_dev, const void *blob_dev, const w12_info *info, uint16_t *y_dev, int M,
                     void *stream) {
    return guarded([&](std::string &err) {
        int rc = check_info(info, err);
        if (rc != W12_OK) return rc;
        if (!x_dev || !blob_dev || !y_dev) {
            err = "null device pointer";
            return (int)W12_ERR_INVALID_ARG;
        }
        if (M < 1 || M > 32) {
            err = "M must be in 1..32";
            return (int)W12_ERR_INVALID_ARG;
        }
        if (!aligned(blob_dev, 256) || !aligned(y_dev, 2) || !aligned(x_dev, 2)) {
            err = "blob_dev must be 256-byte aligned, x_dev and y_dev 2-byte aligned";
            return (int)W12_ERR_ALIGNMENT;
        }
        return w12::launch::gemm_noalloc(x_dev, blob_dev, *info, y_dev, M, stream, &err);
    });
}

int w12_encode_workspace_size(int64_t N, int64_t K, size_t *bytes) {
    return guarded([&](std::string &err) {
        if (!bytes) {
            err = "null pointer";
            return (int)W12_ERR_INVALID_ARG;
        }
        return w12::launch::encode_workspace_size(N, K, bytes, &err);
    });
}

int w12_encoded_size_device(const uint16_t *w_dev, int64_t N, int64_t K, void *workspace, size_t ws_bytes,
                            size_t *bytes, void *stream) {
    return guarded([&](std::string &err) {
        if (!w_dev || !workspace || !bytes) {
            err = "null pointer";
            return (int)W12_ERR_INVALID_ARG;
        }
        if (!aligned(w_dev, 2) || !aligned(workspace, 256)) {
            err = "w_dev must be 2-byte aligned and workspace 256-byte aligned";
            return (int)W12_ERR_ALIGNMENT;
        }
        return w12::launch::encoded_size_device(w_dev, N, K, workspace, ws_bytes, bytes, stream, &err);
    });
}

int w12_encode_device(const uint16_t *w_dev, int64_t N, int64_t K, void *blob_dev, size_t bytes, void *workspace,
                      size_t ws_bytes, void *stream) {
    return guarded([&](std::string &err) {
        if (!w_dev || !blob_dev || !workspace) {
            err = "null device pointer";
            return (int)W12_ERR_INVALID_ARG;
        }
        if (!aligned(w_dev, 2) || !aligned(blob_dev, 256) || !aligned(workspace, 256)) {
            err = "w_dev must be 2-byte aligned, blob_dev and workspace 256-byte aligned";
            return (int)W12_ERR_ALIGNMENT;
        }
        return w12::launch::encode_device(w_dev, N, K, blob_dev, bytes, workspace, ws_bytes, stream, &err);
    });
}

int w12_q8_encoded_size(int64_t N, int64_t K, size_t *bytes) {
    return guarded([&](std::string &err) {
        if (!bytes) {
            err = "null pointer";
            return (int)W12_ERR_INVALID_ARG;
        }
        uint64_t b = 0;
        const int rc = w12::host::q8_encoded_size(N, K, &b, &err);
        if (rc == W12_OK) *bytes = (size_t)b;
        return rc;
    });
}

int w12_q8_encode_host(const uint16_t *w_host, int64_t N, int64_t K, void *blob_host, size_t bytes) {
    return guarded([&](std::string &err) {
        return w12::host::q8_encode(w_host, N, K, static_cast<uint8_t *>(blob_host), bytes, &err);
    });
}

int w12_q8_blob_info(const void *blob_host, size_t bytes, w12_q8_info *out) {
    return guarded([&](std::string &err) {
        return w12::host::q8_parse_header(static_cast<const uint8_t *>(blob_host), bytes, out, &err);
    });
}

int w12_q8_gemm_workspace_size(const w12_q8_info *info, int M, size_t *bytes) {
    return guarded([&](std::string &err) {
        int rc = check_q8_info(info, err);
        if (rc != W12_OK) return rc;
        if (!bytes) {
            err = "null pointer";
            return (int)W12_ERR_INVALID_ARG;
        }
        return w12::launch::q8_workspace_size(*info, M, bytes, &err);
    });
}

int w12_q8_gemm(const uint16_t *x_dev, const void *blob_dev, const w12_q8_info *info, uint16_t *y_dev, int M,
                void *workspace, size_t ws_bytes, void *stream) {
    return guarded([&](std::string &err) {
        int rc = check_q8_info(info, err);
        if (rc != W12_OK) return rc;
        if (!x_dev || !blob_dev || !y_dev || !workspace) {
            err = "null device pointer";
            return (int)W12_ERR_INVALID_ARG;
        }
        if (M < 1 || M > 32) {
            err = "M must be in 1..32";
            return (int)W12_ERR_INVALID_ARG;
        }
        if (!aligned(blob_dev, 256) || !aligned(workspace, 256) || !aligned(y_dev, 2) || !aligned(x_dev, 2)) {
            err = "blob_dev and workspace must be 256-byte aligned, x_dev and y_dev 2-byte aligned";
            return (int)W12_ERR_ALIGNMENT;
        }
        return w12::launch::q8_gemm(x_dev, blob_dev, *info, y_dev, M, workspace, ws_bytes, stream, &err);
    });
}

namespace {
int check_q8_group(int count, const w12_q8_info *infos, std::string &err) {
    if (count < 1 || count > W12_MAX_GROUP || !infos) {
        err = "count must be in 1.." + std::to_string(W12_MAX_GROUP) + " with non-null infos";
        return W12_ERR_INVALID_ARG;
    }
    for (int i = 0; i < count; ++i) {
        const int rc = check_q8_info(&infos[i], err);
        if (rc != W12_OK) return rc;
        if (infos[i].K != infos[0].K) {
            err = "the matrices of a group must share K (they multiply the same x)";
            return W12_ERR_SHAPE;
        }
    }
    return W12_OK;
}
}  // namespace

int w12_q8_gemm_group_launch_info(int count, const w12_q8_info *infos, int M, int32_t out[5]) {
    return guarded([&](std::string &err) {
        int rc = check_q8_group(count, infos, err);
        if (rc != W12_OK) return rc;
        if (!out) {
            err = "out is null";
            return (int)W12_ERR_INVALID_ARG;
        }
        w12::launch::GemmPlan plan;
        rc = w12::launch::q8_group_plan(count, infos, M, &plan, &err);
        if (rc == W12_OK) {
            out[0] = plan.ntok;
            out[1] = plan.splits;
            out[2] = plan.ctas;
            out[3] = plan.ctas_per_sm;
            out[4] = plan.kernel;
        }
        return rc;
    });
}

int w12_q8_gemm_group_workspace_size(int count, const w12_q8_info *infos, int M, size_t *bytes) {
    return guarded([&](std::string &err) {
        int rc = check_q8_group(count, infos, err);
        if (rc != W12_OK) return rc;
        if (!bytes || M < 1 || M > 32) {
            err = "null pointer or M outside 1..32";
            return (int)W12_ERR_INVALID_ARG;
        }
        return w12::launch::q8_group_workspace_size(count, infos, M, bytes, &err);
    });
}

int w12_q8_gemm_group(const uint16_t *x_dev, int count, const void *const *blobs_dev, const w12_q8_info *infos,
                      uint16_t *const *y_devs, int M, void *workspace, size_t ws_bytes, void *stream) {
    return guarded([&](std::string &err) {
        int rc = check_q8_group(count, infos, err);
        if (rc != W12_OK) return rc;
        if (!x_dev || !blobs_dev || !y_devs || !workspace) {
            err = "null pointer";
            return (int)W12_ERR_INVALID_ARG;
        }
        if (M < 1 || M > 32) {
            err = "M must be in 1..32";
            return (int)W12_ERR_INVALID_ARG;
        }
        if (!aligned(workspace, 256) || !aligned(x_dev, 2)) {
            err = "workspace must be 256-byte aligned and x_dev 2-byte aligned";
            return (int)W12_ERR_ALIGNMENT;
        }
        for (int i = 0; i < count; ++i) {
            if (!blobs_dev[i] || !y_devs[i]) {
                err = "null blob or output";
                return (int)W12_ERR_INVALID_ARG;
            }
            if (!aligned(blobs_dev[i], 256) || !aligned(y_devs[i], 2)) {
                err = "each blob must be 256-byte aligned and each y 2-byte aligned";
                return (int)W12_ERR_ALIGNMENT;
            }
        }
        return w12::launch::q8_gemm_group(x_dev, count, blobs_dev, infos, y_devs, M, workspace, ws_bytes, stream,
                                          &err);
    });
}

int w12_read_stream(const void *buf_dev, size_t bytes, void *sink_dev, uint32_t never, void *stream) {
    return guarded([&](std::string &err) {
        if (!buf_dev || !sink_dev) {
            err = "null pointer";
            return (int)W12_ERR_INVALID_ARG;
        }
        if (!aligned(buf_dev, 16) || !aligned(sink_dev, 4) || bytes % 16 != 0) {
            err = "buf_dev must be 16-byte aligned, bytes a multiple of 16, sink_dev 4-byte aligned";
            return (int)W12_ERR_ALIGNMENT;
        }
        return w12::launch::read_stream(buf_dev, bytes, sink_dev, never, stream, &err);
    });
}

int w12_check_status(void *stream) {
    return guarded([&](std::string &err) { return w12::launch::check_status(stream, &err); });
}

int w12_set_option(const char *name, int64_t value) {
    return guarded([&](std::string &err) {
        if (!name) {
            err = "name is null";
            return (int)W12_ERR_INVALID_ARG;
        }
        return w12::launch::set_option(name, value, &err);
    });
}

int w12_get_option(const char *name, int64_t *value) {
    return guarded([&](std::string &err) {
        if (!name || !value) {
            err = "name or value is null";
            return (int)W12_ERR_INVALID_ARG;
        }
        return w12::launch::get_option(name, value, &err);
    });
}

int w12_selftest_timeout(uint32_t timeout_us, void *stream) {
    return guarded([&](std::string &err) { return w12::launch::selftest_timeout(timeout_us, stream, &err); });
}

}  // extern "C"
