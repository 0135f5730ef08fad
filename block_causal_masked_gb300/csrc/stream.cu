// stream.cu -- the streaming cache's new-frame insertion on sm_103a.
//
// FlashDrive tutorial, "流式推理": only the newest camera frame is encoded; its
// pre-RoPE keys and values go into each view's own frame slot of the view-major
// cache (slot `slot` of view w = rows [(w * frames + slot) * per_frame, +
// per_frame)), and its positions into the cache's position array, which the
// attention uses for RoPE and for the streaming mask.  An HBM copy: one thread
// per 16-byte chunk of a (token, KV head) row of K and of V.
#include <cstdint>

#include "launch.h"
#include "ptx.cuh"

namespace bd {
namespace {

__global__ void __launch_bounds__(256) stream_insert_kernel(const __grid_constant__ StreamInsertParams p) {
  pdl_wait();     // the new frame's K/V may come from the previous kernel in the stream
  pdl_trigger();
  const int chunks = p.D / 8;  // 16-byte chunks of a row
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long total = static_cast<long long>(p.views) * p.per_frame * p.Hkv * chunks;
  if (i >= total) return;
  const int c = static_cast<int>(i % chunks);
  const long long r = i / chunks;
  const int h = static_cast<int>(r % p.Hkv);
  const int tok = static_cast<int>(r / p.Hkv);  // w * per_frame + t
  const int w = tok / p.per_frame;
  const int t = tok - w * p.per_frame;
  const long long dst_row = (static_cast<long long>(w) * p.frames + p.slot) * p.per_frame + t;
  const size_t src = (static_cast<size_t>(tok) * p.Hkv + h) * p.D + c * 8;
  const size_t dst = (static_cast<size_t>(h) * p.stride + dst_row) * p.D + c * 8;
  const uint4 kx = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.new_k) + src));
  const uint4 vx = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.new_v) + src));
  *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.k_cache) + dst) = kx;
  *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.v_cache) + dst) = vx;
  if (h == 0 && c == 0) p.k_pos[dst_row] = __ldg(p.new_pos + tok);
}

}  // namespace

cudaError_t launch_stream_insert(const StreamInsertParams& p, cudaStream_t stream) {
  const long long total = static_cast<long long>(p.views) * p.per_frame * p.Hkv * (p.D / 8);
  if (total == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(static_cast<unsigned>((total + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, stream_insert_kernel, p);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace bd
