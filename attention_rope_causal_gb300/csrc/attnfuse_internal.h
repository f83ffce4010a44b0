// Declarations shared by the library's translation units (not part of the public C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "attnfuse.h"
#include "rope.cuh"

namespace attnfuse {

// ---- per-device one-time set-up ----------------------------------------------------------------

// A kernel's set-up on a device (function attributes, SM count) runs once per device and its
// result (an int, e.g. the SM count) is kept.  Safe when several host threads make their first call
// at once: the first runs the set-up under a lock, the others wait for it, and later calls read the
// kept value without locking.  A set-up that fails is tried again on the next call.
class DeviceOnce {
 public:
  static constexpr int kMaxDevices = 64;

  template <typename F>
  cudaError_t get(int dev, F&& setup, int* out) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (done_[dev].load(std::memory_order_acquire)) {
      *out = value_[dev];
      return cudaSuccess;
    }
    std::lock_guard<std::mutex> lock(mu_);
    if (!done_[dev].load(std::memory_order_relaxed)) {
      int v = 0;
      const cudaError_t e = setup(&v);
      if (e != cudaSuccess) return e;
      value_[dev] = v;
      done_[dev].store(true, std::memory_order_release);
    }
    *out = value_[dev];
    return cudaSuccess;
  }

 private:
  std::mutex mu_;
  std::atomic<bool> done_[kMaxDevices] = {};
  int value_[kMaxDevices] = {};
};

// ---- pre-rotation kernel --------------------------------------------------------------------

constexpr int kHeadsPerGroup = 8;

struct RopeJob {
  const void* x;  // [B, N, H, d]
  void* y;        // [B, N, H, d], may equal x
  int H;
  int groups;     // ceil(H / kHeadsPerGroup)
};

struct RopeApplyParams {
  RopeJob job[2];
  int njobs;
  int N;
  long long tokens;  // B * N
  const int32_t* pos;  // [B, N] rotation position of each token (one job only), or nullptr:
  int pos_off;         //   then the position of token (b, n) is pos_off + n
  int pos_neg;         // 1: rotate by the negated position (R^T, the transpose of the rotation)
  int groups_total;  // job[0].groups + (njobs > 1 ? job[1].groups : 0)
  int rot_chunks;    // rotary_dim / 16: item ck < rot_chunks rotates (frequencies 8 ck .. 8 ck + 7)
  int interleaved;   // 0: pairs (k, k + rotary_dim/2); 1: pairs (2k, 2k + 1)
  RopeFreqs freqs;   // F_k for k < rotary_dim / 2
};

cudaError_t launch_rope_apply(const RopeApplyParams& p, int d, bool bf16, cudaStream_t stream);

// ---- attention kernel -----------------------------------------------------------------------

struct AttnParams {
  int B, Hq, Hkv, N;  // N = query rows per batch entry
  int Nk;             // key/value rows per batch entry (>= N)
  int q_off;          // Nk - N: query i is token q_off + i and sees keys j <= q_off + i
  const int32_t* qpos;  // [B, N] query rotation positions, or nullptr (q_off + i)
  const int32_t* kpos;  // [B, Nk] key rotation positions, or nullptr (j)
  int head_pairs;    // 1: a work unit is two query heads of one KV group on the same 128 rows
                     // (Hq / Hkv even); 0: two consecutive 128-row tiles of one head
  int n_qblocks;     // query blocks per head: ceil(N / 128) with head pairs, ceil(N / 256) without
  int total_units;   // B * Hq * n_qblocks, halved with head pairs
  void* out;         // [B, N, Hq, d]  (q is [B, N, Hq, d]; k, v are [B, Nk, Hkv, d])
  float* lse;        // [B, Hq, N] or nullptr
  float scale_log2;  // log2(e) / sqrt(d)
  int rot_chunks;    // rotary_dim / 16 (fused mode: rotation thread chunk ck < rot_chunks works)
  int after_rope_pass;  // 1: launched right after this library's pre-rotation pass on the same stream
  int interleaved;   // 0: pairs (k, k + rotary_dim/2); 1: pairs (2k, 2k + 1)
  unsigned long long timeout_ns;  // limit on any single barrier wait
  RopeFreqs freqs;
};

struct AttnMaps {
  CUtensorMap q, k, v;
};

// Launches the attention kernel.  rotate_q / rotate_k rotate the Q / K tiles on chip (fused mode:
// both; split mode: Q only, K pre-rotated; pre-rotate mode: neither).
cudaError_t launch_attn_fwd(const AttnMaps& maps, const AttnParams& p, int d, bool bf16, bool rotate_q,
                            bool rotate_k, cudaStream_t stream, const char** why);

// ---- decode kernels (few queries, many keys) ---------------------------------------------------

constexpr int kDecodeMaxRows = 16;  // query rows per KV head: (Hq / Hkv) * N

// Decode CTAs resident per SM, warps per CTA and 16-key shared-memory stages per warp: the kernel's
// launch bounds and the key-slice planner both follow them.  At d = 128 one CTA per SM of eight
// warps with three stages each, or -- the 8-row form (at most 8 query rows per KV head) with more
// than 16 (batch, KV head) pairs -- twelve warps with two stages each (its 168 registers a thread
// let twelve warps share the register file; 192 KB of rings either way); at d = 64 two CTAs of
// eight warps with three stages (96 KB each).  With at most 16 pairs (one wave of CTAs, long
// slices) the deeper rings of eight warps measured faster; with more, the extra warps.
constexpr int decode_ctas_per_sm(int d) { return d == 64 ? 2 : 1; }
__host__ __device__ constexpr int decode_stages(int warps) { return warps == 12 ? 2 : 3; }
constexpr int decode_warps(int B, int Hkv, int d, int rows) {
  return d == 128 && rows <= 8 && (long long)B * Hkv > 16 ? 12 : 8;
}
constexpr int kDecodeChunk = 16;  // keys per TMA box and per step of a decode warp

struct DecodeParams {
  const void* q;          // [B, N, Hq, d]
  const void* k;          // [B, Nk, Hkv, d]
  const void* v;          // [B, Nk, Hkv, d]
  void* out;              // [B, N, Hq, d]
  float* lse;             // [B, Hq, N] or nullptr
  int B, Hq, Hkv, N, Nk, q_off;
  const int32_t* qpos;    // [B, N] or nullptr (q_off + i)
  const int32_t* kpos;    // [B, Nk] or nullptr (j)
  int rot_chunks;         // rotary_dim / 16
  int interleaved;
  int keys_per_split;     // multiple of kDecodeChunk
  int n_splits;
  int warps;              // decode_warps(B, Hkv, d, rows): the kernel form the planner assumed
  float scale_log2;       // log2(e) / sqrt(d)
  float* part_o;          // [B, Hkv, n_splits, rows, d] unnormalised partial outputs
  float* part_ml;         // [B, Hkv, n_splits, rows, 2]: running max (log2 units) and sum
  RopeFreqs freqs;
};

struct DecodeMaps {
  CUtensorMap k, v;  // [B, Nk, Hkv, d] in boxes of 64 columns x kDecodeChunk rows, 128-byte swizzle
};

// Split-KV decode: one CTA per (split, KV head, batch) writes partials, a second kernel merges them.
cudaError_t launch_attn_decode(const DecodeMaps& maps, const DecodeParams& p, int d, bool bf16, cudaStream_t stream);

// Reads and clears the decode kernels' device status word (call after synchronising).
cudaError_t read_and_clear_decode_status(unsigned int* value);

// ---- backward kernels ------------------------------------------------------------------------

struct AttnBwdParams {
  int B, Hq, Hkv, N;
  int Nk;                 // key/value rows per batch entry (>= N); the queries are the last N
  int q_off;              // Nk - N: query row i is token q_off + i and sees keys j <= q_off + i
  int n_tiles;            // ceil(N / 128): query tiles
  int n_ktiles;           // ceil(Nk / 128): key tiles
  const void* out;        // [B, N, Hq, d] forward output
  const void* dout;       // [B, N, Hq, d] dL/dout
  const float* lse;       // [B, Hq, N] forward log-sum-exp (natural log)
  float* Dvec;            // [B, Hq, N] workspace: dout . out per row
  void* dq;               // [B, N, Hq, d]
  void* dk;               // [B, Nk, Hkv, d]
  void* dv;               // [B, Nk, Hkv, d]
  float scale_log2;       // log2(e) / sqrt(d)
  float inv_sqrt_d;
  int unrotate;           // 1: the epilogues apply R^T (half-split over all d, positions q_off + i and j);
                          // 0: they write the gradients in the rotated frame (a pass rotates back)
  unsigned long long timeout_ns;
  int* unit_ctr;          // workspace: next unit of the dQ kernel (zeroed by the D kernel)
  RopeFreqs freqs;        // F_k, k < d/2 (half-split, rotary dimension d)
};

struct AttnBwdMaps {
  CUtensorMap q, k, v, dout;          // q, k: the rotated copies; boxes of 128 rows
  CUtensorMap q64, k64, v64, dout64;  // the same tensors in boxes of 64 rows (the streamed tiles)
};

// Launches D = rowsum(dout * out), then the dK/dV and dQ kernels (rotated q, k already in place).
cudaError_t launch_attn_bwd(const AttnBwdMaps& maps, const AttnBwdParams& p, int d, bool bf16, cudaStream_t stream);

// Reads and clears the backward kernels' device status word (call after synchronising).
cudaError_t read_and_clear_bwd_status(unsigned int* value);

// Device status word written by kernels whose barrier waits ran out (bit 0).
cudaError_t read_and_clear_device_status(unsigned int* value, cudaStream_t stream);

// Launches one CTA that waits, for at most timeout_ns, on a barrier nothing arrives on.
cudaError_t launch_diag_wait_timeout(unsigned long long timeout_ns, cudaStream_t stream);

// Fills F_k = round(theta_k / (2 pi) * 2^64), theta_k = base^(-2k/r), k < r/2 (r = rotary dimension).
void rope_freqs_host(int r, double base, RopeFreqs* f);

// Sets the calling thread's attnfuse_last_error() message (printf-style).
void set_last_error(const char* fmt, ...);

// The argument checks of attnfuse_rope_causal_fwd (pointers, sizes, alignment, mode, dtype, head
// dimension, base) and the device check (sm_103), in that order; no device work.
attnfuse_status_t check_fwd_call(const void* q, const void* k, const void* v, const void* out, const float* lse, int B,
                                 int Hq, int Hkv, int N, int d, double rope_base, attnfuse_mode_t mode,
                                 attnfuse_dtype_t dtype);

}  // namespace attnfuse
