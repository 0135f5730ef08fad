// launch.h -- internal host-side interface between the C ABI (api.cu) and the
// kernels (attn.cu, vocab.cu).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

namespace bd {

// Runs a set-up step once per device -- kernel attributes such as the dynamic
// shared-memory limit belong to the device that is current when they are set
// -- and again on a device where it failed.  Thread-safe.
class PerDeviceOnce {
 public:
  template <typename F>
  cudaError_t run(F&& setup) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu_);
    if (done_[dev]) return cudaSuccess;
    e = setup();
    if (e == cudaSuccess) done_[dev] = true;
    return e;
  }

 private:
  static constexpr int kMaxDevices = 64;
  std::mutex mu_;
  bool done_[kMaxDevices] = {};
};

constexpr int kAttnBM = 128;        // packed query rows per CTA (tcgen05 M)
constexpr int kAttnBN = 128;        // keys per K/V tile
constexpr int kAttnMaxTiles = 4096; // K/V tiles of one (row tile, KV head) before splitting
constexpr int kAttnMaxSplits = 16;  // KV splits = CTAs of one cluster

// Clusters of S attention CTAs (one CTA per SM: ~200 KB of shared memory and
// all 512 TMEM columns) that a full GB300 holds at once, as
// cudaOccupancyMaxActiveClusters reports it for 1 <= S <= 16: the GPCs fit
// fewer wide clusters than 152 / S.  Used when no device can be asked.
__host__ __device__ constexpr int attn_resident_clusters(int S) {
  constexpr int kTable[17] = {0, 152, 76, 46, 36, 28, 23, 15, 15, 15, 13, 8, 8, 7, 7, 7, 7};
  return S >= 1 && S <= 16 ? kTable[S] : 0;
}

// Split-KV merge: CTA q of a cluster of S merges packed rows [q * r, (q + 1) * r)
// of the tile, r = ceil(128 / S) rounded up to even.
__host__ __device__ constexpr int attn_merge_rows(int S) { return ((kAttnBM + S - 1) / S + 1) & ~1; }
// Partial O of one (KV head, row tile) in the slices that one split hands one
// owner: [S owners][S splits][D / 8][r] bf16x8 chunks of the splits'
// normalised O, so that an owner's slices are one contiguous range.  (The splits' running max and sum travel through
// distributed shared memory.)
__host__ __device__ constexpr long long attn_part_bytes(int S, int D) {
  return static_cast<long long>(S) * S * attn_merge_rows(S) * 2 * D;
}

// Everything the attention kernels need, in the fork's terms: plain attention is
// the fork with N = 1, the prefix = rows [0, C) of K/V and the private rows =
// the active rows [C, C + n_q) (priv_len = 0).
struct AttnParams {
  const void* q;          // bf16 [N, n_q, Hq, D]
  void* o;                // bf16 [N, n_q, Hq, D]
  float* lse;             // fp32 [N, Hq, n_q] or null
  void* part;             // split partials (splits > 1): [Hkv, m_tiles] blocks of attn_part_bytes
  int m_tiles;            // row tiles per KV head (all launches of the call)
  int m_tile0;            // first row tile of this launch (grid y counts from here)
  const int32_t* block_start;  // [n_blocks + 1] or null (uniform block_size)
  int32_t* dev_status;
  int N, n_q, Hq, Hkv, G, D, C, priv_len, n_blocks, block_size, num_splits;
  int rows_per_head;      // N * n_q * G
  int n_prefix_tiles;     // ceil(C / BN)
  float scale_log2;       // sm_scale * log2(e)
  int q_tma;              // Q tile by TMA (G divides 128)
  int prefix_early;       // prefix K/V tiles may be loaded before the dependency wait
  // streaming mask (q_pos != null): queries over the prefix only, key j visible
  // iff (kpos ? kpos[j] : j) - kdelta <= q_pos[i]
  const int32_t* q_pos;
  const int32_t* kpos;
  int kdelta;
  unsigned long long wait_ns;  // limit of a pipeline wait (drains keep the full limit)
  // FP8 (E4M3) K/V (kv8 != 0): the tiles arrive as bytes and are dequantised to
  // fp16 in shared memory; row r of a segment is scaled by 2^exp[., (row0 + r) / 128]
  int kv8;
  const int8_t* pk_exp;   // prefix [Hkv, p_exp_stride]
  const int8_t* pv_exp;
  const int8_t* rk_exp;   // private [N, Hkv, r_exp_stride]
  const int8_t* rv_exp;
  int p_exp_stride, r_exp_stride, r_exp_row0;
};

// New frame of the streaming cache written into every view's frame slot.
struct StreamInsertParams {
  void* k_cache;          // bf16 [Hkv, stride, D]
  void* v_cache;
  int32_t* k_pos;         // [views * frames * per_frame]
  const void* new_k;      // bf16 [views * per_frame, Hkv, D]
  const void* new_v;
  const int32_t* new_pos; // [views * per_frame]
  int views, frames, per_frame, slot, Hkv, D;
  long long stride;
};

// Rotation of the cached prefix keys before attention (RoPE at k_pos - delta).
struct RopeParams {
  const void* k;          // bf16 [Hkv, stride, D], rows [0, C) rotated
  void* out;              // bf16 [Hkv, C, D]
  const int32_t* k_pos;   // [C] or null (position = key index)
  int Hkv, C, D, delta;
  long long stride;
  unsigned long long turns[64];  // theta^(-2d/D) / (2*pi) as a 0.64 fixed-point fraction
  double freq[64];               // theta^(-2d/D) in float64
  float two_pi_64[2];            // 2 pi / 2^64 as float-float
};

struct AttnMaps {
  CUtensorMap q;          // Q: 4D (D, G, Hkv, N * n_q), box {64, G, 1, 128 / G}
  CUtensorMap pk, pv;     // prefix K/V: 3D (D, C, Hkv); bf16 box {64, 128, 1}, or E4M3 box {D, 128, 1}
  CUtensorMap rk, rv;     // private K/V: 4D (D, priv_len + n_q, Hkv, N)
};

int attn_smem_bytes(int D, bool kv8);
// Clusters of S attention CTAs (head dim D) the current device holds at once
// (cudaOccupancyMaxActiveClusters, cached per device), or the full-GB300
// table when no device answers.
int attn_max_clusters(int S, int D);
cudaError_t launch_attention(const AttnParams& p, const AttnMaps& maps, int m_tiles, cudaStream_t stream);
cudaError_t launch_rope_prefix(const RopeParams& p, cudaStream_t stream);
cudaError_t launch_stream_insert(const StreamInsertParams& p, cudaStream_t stream);

// ---------------------------------------------------------------- vocab reductions

struct UnmaskParams {
  const void* logits;
  int dtype;              // 0 f32, 1 bf16
  long long ld;
  int R, V;
  const int32_t* logit_row;
  int n_pos;
  const int32_t* block_start;
  int n_blocks;
  uint8_t* state;
  int32_t* tokens;
  float tau_full, tau_half;
  int min_num, min_den, k_fixed, add_num, add_den, act_num, act_den;
  uint8_t* commit;
  int32_t* n_committed;
  int32_t* status;
  int32_t* pred;
  float* conf;
  float* lse;
  int write_draft;
  int32_t* dev_status;
  unsigned long long wait_ns;  // limit of a wait for a streamed piece
  // workspace carve-up
  float4* row_res;            // [R]: (max, sum of exp(l - max), argmax bits, -) of each row
  unsigned int* grid_ticket;  // [1]
  int chunks;                 // CTAs per logits row (one cluster)
  int chunk_elems;            // elements per chunk (multiple of 8)
};

struct VerifyParams {
  int n_seq, L;
  int32_t* tokens;
  uint8_t* state;
  const void* logits;
  int dtype;
  long long ld;
  int n_rows, V;
  const float* noise;
  float inv_temp;
  int32_t* accepted_len;
  int32_t* bonus;
  int32_t* bonus_pos;
  int32_t* dev_status;
  unsigned long long wait_ns;
  float4* row_res;            // [n_seq * n_rows]: (best score, -, argmax bits, -) of each row
  unsigned int* seq_ticket;   // [n_seq]
  int chunks;
  int chunk_elems;
};

constexpr int kMaxPos = 2048;          // positions of one unmask window
constexpr int kMaxChunks = 16;         // CTAs (chunks) of one logits row = one thread-block cluster
constexpr int kMaxVerifyRows = 65535;  // n_seq * n_rows of one verify call (grid y)
constexpr int kMaxVerifySeqs = 1024;   // sequences of one verify call

size_t unmask_counter_bytes();
size_t verify_counter_bytes();
size_t unmask_workspace_bytes(int R);
size_t verify_workspace_bytes(int n_seq, int n_rows);
void vocab_split(int rows, int V, int num_sms, int* chunks, int* chunk_elems, int max_chunks = kMaxChunks);
cudaError_t launch_unmask(const UnmaskParams& p, cudaStream_t stream);
cudaError_t launch_verify(const VerifyParams& p, cudaStream_t stream);

}  // namespace bd
