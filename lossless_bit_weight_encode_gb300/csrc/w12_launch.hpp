// Launch layer between the C ABI (capi.cpp) and the CUDA kernels (kernels.cu).
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>

#include "w12.h"

namespace w12 {
namespace launch {

// How w12_gemm will run a problem on the current device.
struct GemmPlan {
    bool gemv = false;      // one token on CUDA cores instead of tensor cores
    bool gemv_sm = false;   // the CUDA-core kernel with one CTA per SM
    bool tc_sm = false;     // the tensor-core kernel with one CTA per SM
    int ntok = 16;          // MMA token width (16 or 32)
    int splits = 1;         // CTAs per tile along K (stream-K: the most CTAs sharing a tile)
    int ctas = 0;           // grid size
    int64_t units = 0;      // stream-K: tiles x segments shared by the ctas (0: fixed split-K)
    int ctas_per_sm = 0;    // resident CTAs per SM the plan assumed
    int kernel = 0;         // W12_KERNEL_* of include/w12.h
    size_t ws_counters = 0, ws_partials = 0, ws_x = 0;  // workspace offsets
    size_t ws_bytes = 0;
};

int plan_gemm(const w12_info &info, int M, GemmPlan *plan, std::string *err, bool q8 = false);

int group_plan(int count, const w12_info *infos, int M, GemmPlan *plan, std::string *err);

int q8_workspace_size(const w12_q8_info &info, int M, size_t *bytes, std::string *err);

int q8_gemm(const uint16_t *x_dev, const void *blob_dev, const w12_q8_info &info, uint16_t *y_dev, int M,
            void *workspace, size_t ws_bytes, void *stream, std::string *err);

int q8_group_plan(int count, const w12_q8_info *infos, int M, GemmPlan *plan, std::string *err);

int q8_group_workspace_size(int count, const w12_q8_info *infos, int M, size_t *bytes, std::string *err);

int q8_gemm_group(const uint16_t *x_dev, int count, const void *const *blobs, const w12_q8_info *infos,
                  uint16_t *const *ys, int M, void *workspace, size_t ws_bytes, void *stream, std::string *err);

int decode(const void *blob_dev, const w12_info &info, uint16_t *out_dev, void *stream, std::string *err);

int read_stream(const void *buf_dev, size_t bytes, void *sink_dev, uint32_t never, void *stream, std::string *err);

int gemm(const uint16_t *x_dev, const void *blob_dev, const w12_info &info, uint16_t *y_dev, int M,
         void *workspace, size_t ws_bytes, void *stream, std::string *err);

int group_workspace_size(int count, const w12_info *infos, int M, size_t *bytes, std::string *err);

int gemm_group(const uint16_t *x_dev, int count, const void *const *blobs, const w12_info *infos,
               uint16_t *const *ys, int M, void *workspace, size_t ws_bytes, void *stream, std::string *err);

int argmax_workspace_size(const w12_info &info, int M, size_t *bytes, std::string *err);

int gemm_argmax(const uint16_t *x_dev, const void *blob_dev, const w12_info &info, int M, uint16_t *y_dev,
                int32_t *idx_dev, float *val_dev, void *workspace, size_t ws_bytes, void *stream, std::string *err);

int gemm_noalloc(const uint16_t *x_dev, const void *blob_dev, const w12_info &info, uint16_t *y_dev, int M,
                 void *stream, std::string *err);

int check_status(void *stream, std::string *err);

int encode_workspace_size(int64_t N, int64_t K, size_t *bytes, std::string *err);

int encoded_size_device(const uint16_t *w_dev, int64_t N, int64_t K, void *workspace, size_t ws_bytes,
                        size_t *bytes, void *stream, std::string *err);

int encode_device(const uint16_t *w_dev, int64_t N, int64_t K, void *blob_dev, size_t cap, void *workspace,
                  size_t ws_bytes, void *stream, std::string *err);

int selftest_timeout(uint32_t timeout_us, void *stream, std::string *err);

int set_option(const char *name, int64_t value, std::string *err);
int get_option(const char *name, int64_t *value, std::string *err);

}  // namespace launch
}  // namespace w12
