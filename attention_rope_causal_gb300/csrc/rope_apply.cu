// Pre-rotation pass: applies RoPE to Q and K in HBM (out of place or in place) before a plain
// causal attention kernel runs on the rotated tensors.  This is the "separate operation" the
// AttnFuse report weighs against in-kernel rotation ("AttnFuse Makes RoPE a First-Class Attention
// Compilation Operation", 2026-09-13 AI papers report, paragraphs 3-5: pre-rotation costs memory
// bandwidth, fused rotation costs compute).
//
// It is an elementwise stream, bounded by HBM bandwidth: every element is read once and written
// once.  Work item = (token, head group of up to kHeadsPerGroup heads, item index ck < d/16), each
// item two 16-byte chunks of a head row.  Consecutive threads cover contiguous 16-byte chunks, so
// each warp-wide 16-byte load or store touches whole 128-byte segments.  A thread computes the
// cos/sin of its 8 frequencies once and applies them to every head of its group, keeping 4 heads
// (8 loads of 16 bytes) in flight.  RoPE variants: only the first rotary_dim entries rotate (the
// rest are copied), in half-split or interleaved pairs.  The rotation position of token (b, n) is
// read from a per-token array, or is a fixed offset plus n.
#include <cuda_runtime.h>

#include "attnfuse_internal.h"
#include "rope.cuh"

namespace attnfuse {

namespace {

constexpr int kThreads = 256;

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads) rope_apply_kernel(const __grid_constant__ RopeApplyParams p) {
  constexpr int NCH = D / 16;  // work items per head row; each covers two 16-byte chunks
  ptx::grid_dep_launch_dependents();  // the attention kernel after this pass may start its prologue
  const long long item = (long long)blockIdx.x * kThreads + threadIdx.x;
  const long long per_token = (long long)p.groups_total * NCH;
  const long long token = item / per_token;
  if (token >= p.tokens) return;
  const int rem = (int)(item - token * per_token);
  int g = rem / NCH;
  const int ck = rem - g * NCH;
  const int32_t pos0 = p.pos ? p.pos[token] : p.pos_off + (int32_t)(token % p.N);
  const int32_t pos = p.pos_neg ? -pos0 : pos0;

  int j = 0;
  if (g >= p.job[0].groups) {
    g -= p.job[0].groups;
    j = 1;
  }
  const RopeJob jb = p.job[j];
  const int h0 = g * kHeadsPerGroup;
  const int nh = min(kHeadsPerGroup, jb.H - h0);

  // Chunks (16 bytes = 8 elements) of a row: the first 2R = rotary_dim / 8 are rotated.  Item ck < R
  // rotates, with frequencies 8 ck .. 8 ck + 7, either chunks ck and ck + R (pairs (k, k + r/2)) or
  // the adjacent chunks 2 ck, 2 ck + 1 (pairs (2k, 2k + 1)).  Items ck >= R copy chunks 2 ck and
  // 2 ck + 1 when the output is not the input.
  const int R = p.rot_chunks;
  const bool rotate = ck < R;
  if (!rotate && jb.x == jb.y) return;
  const int ca = rotate && !p.interleaved ? ck : 2 * ck;
  const int cb = rotate && !p.interleaved ? ck + R : 2 * ck + 1;

  float c[8], s[8];
  if (rotate) {
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int k = ck * 8 + t;
      rope_cs_signed(pos, p.freqs.lo[k], p.freqs.hi[k], c[t], s[t]);
    }
  }

  const size_t row_bytes = (size_t)D * 2;
  const size_t off0 = ((size_t)token * jb.H + h0) * row_bytes;
  const char* xb = reinterpret_cast<const char*>(jb.x) + off0;
  char* yb = reinterpret_cast<char*>(jb.y) + off0;

  for (int h = 0; h < nh; h += 4) {
    uint4 av[4], bv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (h + u < nh) {
        av[u] = __ldg(reinterpret_cast<const uint4*>(xb + (size_t)(h + u) * row_bytes + ca * 16));
        bv[u] = __ldg(reinterpret_cast<const uint4*>(xb + (size_t)(h + u) * row_bytes + cb * 16));
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (h + u < nh) {
        if (rotate) {
          if (p.interleaved) {
            rope_rotate_chunk_il<BF16>(av[u], c, s);
            rope_rotate_chunk_il<BF16>(bv[u], c + 4, s + 4);
          } else {
            rope_rotate_chunk<BF16>(av[u], bv[u], c, s);
          }
        }
        *reinterpret_cast<uint4*>(yb + (size_t)(h + u) * row_bytes + ca * 16) = av[u];
        *reinterpret_cast<uint4*>(yb + (size_t)(h + u) * row_bytes + cb * 16) = bv[u];
      }
    }
  }
}

}  // namespace

cudaError_t launch_rope_apply(const RopeApplyParams& p, int d, bool bf16, cudaStream_t stream) {
  const int nch = d / 16;
  const long long items = p.tokens * (long long)p.groups_total * nch;
  if (items <= 0) return cudaSuccess;
  const long long blocks = (items + kThreads - 1) / kThreads;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)blocks), block(kThreads);
  if (d == 128) {
    if (bf16)
      rope_apply_kernel<128, true><<<grid, block, 0, stream>>>(p);
    else
      rope_apply_kernel<128, false><<<grid, block, 0, stream>>>(p);
  } else {
    if (bf16)
      rope_apply_kernel<64, true><<<grid, block, 0, stream>>>(p);
    else
      rope_apply_kernel<64, false><<<grid, block, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace attnfuse
