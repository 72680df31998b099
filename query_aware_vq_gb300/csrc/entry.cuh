// entry.cuh -- argument checks shared by the extern "C" entry points (defined
// in api.cu), so that every entry point validates a shape, a dtype, a
// fraction or the RoPE parameters the same way.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/a2ats.h"
#include "common.cuh"

namespace a2ats {

bool dtype_ok(int32_t dt);
// d multiple of 8 in [8, 256]; positions below 2^24 (exact in fp32);
// B <= 2^20, H <= 4096, B*H <= 65535.
int check_shape(int64_t B, int64_t H, int64_t Ncap, int64_t d);
bool unit_interval(double v);  // false for NaN
// Fill the device-side RoPE constants; enabled = 0 when p is null.
int make_rope(const a2ats_rope_params* p, int64_t d, RopeArgs& ra);
// Record CUDA's message for a2ats_last_error and return A2ATS_ERR_CUDA.
int cuda_fail(cudaError_t e);

}  // namespace a2ats
