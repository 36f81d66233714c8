// Internal declarations of the decoding kernels over compressed caches (kvc_decode.cu).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvc.h"

namespace kvc {

cudaError_t take_status_decode(unsigned int* v);

// Attention of one new query per head over a cache whose keys keep Ck = kd.D channels.
// Splits each (b, kvh) row's keys over `nsplit` CTAs; partials live in the workspace.
struct DecodePlan {
  int nsplit;         // key ranges per (b, kvh)
  int head_groups;    // CTAs per key range along the query group (16 heads each)
  int64_t chunks;     // 16-key chunks per row
  size_t part_bytes;  // workspace: o [rows][nsplit][G][D] float + (m, l) [rows][nsplit][G] float2
};
DecodePlan plan_decode(const kvc_kv_desc& vd);
bool decode_shape_supported(int Ck, int D);
cudaError_t launch_decode_attention(const uint16_t* q, const int32_t* ch, const uint16_t* K, const kvc_kv_desc& kd,
                                    const uint16_t* V, const kvc_kv_desc& vd, const uint32_t* live, float scale,
                                    float* out, void* ws, cudaStream_t st);
// K_out[b,kvh,j,ch[c]] = Kp[b,kvh,j,c]; other channels 0
cudaError_t launch_zero_add_back(const uint16_t* Kp, const kvc_kv_desc& pd, const int32_t* ch, uint16_t* Ko,
                                 const kvc_kv_desc& od, cudaStream_t st);

}  // namespace kvc
