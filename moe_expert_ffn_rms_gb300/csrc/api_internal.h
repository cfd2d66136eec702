// Internal helpers of api.cu shared with other entry-point files.
#pragma once

#include "../../include/moe_ffn.h"

namespace moe {

// Records `msg` as this thread's moe_last_error() text and returns `s`.
moe_status api_fail(moe_status s, const char* msg);

// Status of the shape checks moe_ffn_forward applies (MOE_OK if valid).
moe_status api_check_shape(const moe_shape* shape);

}  // namespace moe
