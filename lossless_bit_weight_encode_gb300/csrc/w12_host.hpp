// Host-side pieces of the W12 library: encoder, header parsing, blob checks.
#pragma once

#include <cstdint>
#include <string>

#include "w12.h"
#include "w12_format.hpp"

namespace w12 {
namespace host {

// N, K in [1, 2^31] with every offset far inside 63 bits (the encoders' limit).
bool check_shape(int64_t N, int64_t K, std::string *err);
int encoded_size(const uint16_t *w, int64_t N, int64_t K, uint64_t *bytes, std::string *err);
int encode(const uint16_t *w, int64_t N, int64_t K, uint8_t *blob, uint64_t cap, std::string *err);
int parse_header(const uint8_t *blob, uint64_t bytes, w12_info *out, std::string *err);
int validate(const uint8_t *blob, uint64_t bytes, std::string *err);

int q8_encoded_size(int64_t N, int64_t K, uint64_t *bytes, std::string *err);
int q8_encode(const uint16_t *w, int64_t N, int64_t K, uint8_t *blob, uint64_t cap, std::string *err);
int q8_parse_header(const uint8_t *blob, uint64_t bytes, w12_q8_info *out, std::string *err);

}  // namespace host
}  // namespace w12
