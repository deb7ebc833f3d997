// Internal declarations shared by the host translation units of libqfmt.
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/qfmt.h"

namespace qfmt {

// Record a failure message for qfmt_last_error() and return `status`.
int fail(int status, const char* fmt, ...);
void clear_error();

bool valid_format(int fmt);
int block_of(int fmt);          // 0 for an unknown format
bool is_4bit(int fmt);
int scale_entry_bytes(int fmt);  // bytes per scale entry: 1, 2, 4 (mxfp4x2: 8)
int sub_bits(int fmt);           // 2, 3, 5, 6 for the sub-byte integer formats; 0 otherwise
int code_bits(int fmt);          // bits per code

// Shape/argument checks shared by the device entry points.  Returns QFMT_OK
// or a failure status (message recorded).
int check_group(int fmt, int group);
int check_shape(int fmt, int64_t M, int64_t N, int64_t K);
int check_ptr(const void* p, int align, const char* what);

}  // namespace qfmt
