// Causal RoPE attention for a few queries against many keys (decode, short prefill after a cache):
// split-KV on the CUDA cores.  With N queries and rows = (Hq / Hkv) N <= 16 query rows per KV head
// the tensor-core tile kernels keep one useful row in 128 and take ~25x the HBM time of reading K
// and V; this path reads every K and V row once.
//
// What it computes: the function of attnfuse_rope_causal_fwd (header of include/attnfuse.h) in
// its general form -- the N queries are the last N of the Nk tokens, query i sees keys j <= Nk - N
// + i, rotation positions q_off + i and j or the explicit arrays, any rotary dimension and pairing
// ("AttnFuse Makes RoPE a First-Class Attention Compilation Operation", paragraphs 1-2: RoPE on Q
// and K before the product, causal mask, softmax).
//
// attn_decode_kernel: one CTA per (split of keys_per_split keys, KV head, batch), 256 threads.  The
// CTA rotates its query rows once (exact cos/sin per row) into fp32 shared memory, then walks its
// keys 64 at a time: K and V rows to shared memory (16-byte loads), K rotated there at each key's
// position (exact cos/sin, rounded to the input type like the other paths), scores for every (row,
// key), online softmax per row (exp2, fp32 max and sum), O += P V in registers.  It writes the
// unnormalised O, the running max (log2 units) and the sum of its split.
// attn_decode_combine_kernel: one warp per (batch, KV head, row) merges the splits (rescaling each
// by 2^(m_s - m)) into out and lse.
// No barrier waits, so nothing here can time out.
#include <cuda_runtime.h>
#include <math.h>

#include <type_traits>

#include "attnfuse_internal.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace attnfuse {

namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 64;  // keys per step
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct DecCfg {
  static constexpr int KSTRIDE = D + 8;  // bf16/fp16 elements per K row in shared memory (padding
                                         // spreads consecutive rows over the banks)
  static constexpr uint32_t OFF_Q = 0;                                            // fp32 [rows][D]
  static constexpr uint32_t OFF_K = OFF_Q + kDecodeMaxRows * D * 4;               // 16-bit [64][KSTRIDE]
  static constexpr uint32_t OFF_V = OFF_K + kChunk * KSTRIDE * 2;                 // 16-bit [64][D]
  static constexpr uint32_t OFF_S = OFF_V + kChunk * D * 2;                       // fp32 [rows][64 keys]
  static constexpr uint32_t OFF_ROW = OFF_S + kDecodeMaxRows * kChunk * 4;        // fp32 [rows] m, l, alpha
  static constexpr uint32_t OFF_FREQ = OFF_ROW + 3 * kDecodeMaxRows * 4;         // u32 F_k lo[64], hi[64]
  static constexpr uint32_t SMEM = OFF_FREQ + 2 * 64 * 4;
};

// Offsets, inside a head vector, of the 8 rotation pairs of frequency group fg (frequencies
// 8 fg .. 8 fg + 7): pair t is (a[t], b[t]).  Half-split over the rotary dimension r: (8 fg + t,
// r/2 + 8 fg + t); interleaved: (16 fg + 2t, 16 fg + 2t + 1).
__device__ __forceinline__ void pair_index(int fg, int t, int r, bool interleaved, int& ia, int& ib) {
  if (interleaved) {
    ia = 16 * fg + 2 * t;
    ib = ia + 1;
  } else {
    ia = 8 * fg + t;
    ib = r / 2 + ia;
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads) attn_decode_kernel(const __grid_constant__ DecodeParams p) {
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  using C = DecCfg<D>;
  extern __shared__ __align__(16) uint8_t smem[];
  float* sQ = reinterpret_cast<float*>(smem + C::OFF_Q);
  T* sK = reinterpret_cast<T*>(smem + C::OFF_K);
  T* sV = reinterpret_cast<T*>(smem + C::OFF_V);
  float* sS = reinterpret_cast<float*>(smem + C::OFF_S);
  float* sM = reinterpret_cast<float*>(smem + C::OFF_ROW);
  float* sL = sM + kDecodeMaxRows;
  float* sA = sL + kDecodeMaxRows;
  uint32_t* sF = reinterpret_cast<uint32_t*>(smem + C::OFF_FREQ);  // lo[64] then hi[64]

  const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const int g = p.Hq / p.Hkv;
  const int rows = g * p.N;  // row = local head * N + query index
  const int r = 2 * p.rot_chunks * 8;  // rotary dimension
  const bool il = p.interleaved != 0;
  const int key0 = split * p.keys_per_split;
  const int key_end = min(p.Nk, key0 + p.keys_per_split);

  // ---- query rows, rotated (exact cos/sin per row), scaled into fp32 shared memory ----------
  for (int idx = tid; idx < rows * (D / 8); idx += kThreads) {
    const int row = idx / (D / 8), c8 = idx % (D / 8);
    const int hl = row / p.N, i = row % p.N;
    const T* src = reinterpret_cast<const T*>(p.q) + (((size_t)b * p.N + i) * p.Hq + hk * g + hl) * D + 8 * c8;
    const uint4 w = *reinterpret_cast<const uint4*>(src);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float lo, hi;
      Pack<BF16>::unpack(ws[e], lo, hi);
      sQ[row * D + 8 * c8 + 2 * e] = lo;
      sQ[row * D + 8 * c8 + 2 * e + 1] = hi;
    }
  }
  if (tid < kDecodeMaxRows) {
    sM[tid] = -INFINITY;
    sL[tid] = 0.f;
  }
  // F_k in shared memory: per-lane frequency indices would serialise constant-bank loads.
  if (tid < 64) sF[tid] = p.freqs.lo[tid];
  else if (tid < 128) sF[tid] = p.freqs.hi[tid - 64];
  __syncthreads();
  for (int idx = tid; idx < rows * p.rot_chunks; idx += kThreads) {
    const int row = idx / p.rot_chunks, fg = idx % p.rot_chunks;
    const int i = row % p.N;
    const int32_t pos = p.qpos ? p.qpos[(size_t)b * p.N + i] : p.q_off + i;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      float c, s;
      rope_cs_signed(pos, sF[8 * fg + t], sF[64 + 8 * fg + t], c, s);
      int ia, ib;
      pair_index(fg, t, r, il, ia, ib);
      const float x = sQ[row * D + ia], y = sQ[row * D + ib];
      float xr, yr;
      rope_pair(x, y, c, s, xr, yr);
      // rotated query rounded to the input type once, as in the other paths
      float2 rr;
      Pack<BF16>::unpack(Pack<BF16>::pack(xr, yr), rr.x, rr.y);
      sQ[row * D + ia] = rr.x;
      sQ[row * D + ib] = rr.y;
    }
  }
  // Rows past the rotary dimension and unrotated entries were already exact copies.

  // O accumulators: thread owns items (row, column pair) it = tid + kThreads * n.
  constexpr int kMaxItems = kDecodeMaxRows * (D / 2) / kThreads;  // 4 (d = 128) or 2 (d = 64)
  float oacc[kMaxItems][2];
#pragma unroll
  for (int n = 0; n < kMaxItems; ++n) oacc[n][0] = oacc[n][1] = 0.f;
  const int n_items = rows * (D / 2);

  // K and V rows of a chunk: LPT 16-byte pieces per thread, all loads issued before any is used;
  // the next chunk's are in flight while the current one is computed on.
  constexpr int LPT = kChunk * (D / 8) / kThreads;  // 4 (d = 128) or 2 (d = 64)
  uint4 kpre[LPT], vpre[LPT];
  auto load_chunk = [&](int kc) {
#pragma unroll
    for (int n = 0; n < LPT; ++n) {
      const int idx = tid + kThreads * n, kr = idx / (D / 8), c8 = idx % (D / 8);
      const int j = kc + kr;
      kpre[n] = vpre[n] = make_uint4(0, 0, 0, 0);  // zero past the split or the sequence
      if (j < key_end) {
        const size_t off = (((size_t)b * p.Nk + j) * p.Hkv + hk) * D + 8 * c8;
        kpre[n] = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.k) + off));
        vpre[n] = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.v) + off));
      }
    }
  };
  if (key0 < key_end) load_chunk(key0);
  // cos/sin of the thread's key-rotation items (see below) and their advance by 64 positions.
  constexpr int KIT = (kChunk * (D / 16) + kThreads - 1) / kThreads;  // 2 (d = 128) or 1 (d = 64)
  RopeCS8 kcs[KIT], kstep[KIT];
#pragma unroll
  for (int n = 0; n < KIT; ++n) {
    const int idx = tid + kThreads * n;
    const int fg = p.rot_chunks > 0 ? idx % p.rot_chunks : 0;
    rope_cs8_exact((uint32_t)kChunk, sF, sF + 64, 8 * fg, kstep[n]);
  }

  for (int kc = key0; kc < key_end; kc += kChunk) {
    __syncthreads();  // previous chunk's K, V, S no longer read
#pragma unroll
    for (int n = 0; n < LPT; ++n) {
      const int idx = tid + kThreads * n, kr = idx / (D / 8), c8 = idx % (D / 8);
      *reinterpret_cast<uint4*>(sK + kr * C::KSTRIDE + 8 * c8) = kpre[n];
      *reinterpret_cast<uint4*>(sV + kr * D + 8 * c8) = vpre[n];
    }
    if (kc + kChunk < key_end) load_chunk(kc + kChunk);
    __syncthreads();
    // ---- rotate the chunk's keys in place ------------------------------------------------------
    // Thread item n: key row kr, frequency group fg (8 frequencies, two 16-byte pieces).  Positions
    // j: cos/sin carried from chunk to chunk by the exact rotation of 64 positions, exact again every
    // 16 chunks; explicit positions: exact per key.
#pragma unroll
    for (int n = 0; n < KIT; ++n) {
      const int idx = tid + kThreads * n;
      if (idx >= kChunk * p.rot_chunks) break;
      const int kr = idx / p.rot_chunks, fg = idx % p.rot_chunks;
      const int j = kc + kr;
      if (p.kpos != nullptr) {
        if (j < key_end) rope_cs8_exact_signed(p.kpos[(size_t)b * p.Nk + j], sF, sF + 64, 8 * fg, kcs[n]);
      } else if (((kc - key0) / kChunk) % 16 == 0) {
        rope_cs8_exact((uint32_t)j, sF, sF + 64, 8 * fg, kcs[n]);
      }
      if (j < key_end) {
        T* row = sK + kr * C::KSTRIDE;
        if (il) {
          uint4* a = reinterpret_cast<uint4*>(row + 16 * fg);
          uint4 x = a[0], y = a[1];
          rope_rotate_chunk_il_cs8<BF16>(x, kcs[n], 0);
          rope_rotate_chunk_il_cs8<BF16>(y, kcs[n], 1);
          a[0] = x;
          a[1] = y;
        } else {
          uint4* xa = reinterpret_cast<uint4*>(row + 8 * fg);
          uint4* ya = reinterpret_cast<uint4*>(row + r / 2 + 8 * fg);
          uint4 x = *xa, y = *ya;
          rope_rotate_chunk_cs8<BF16>(x, y, kcs[n]);
          *xa = x;
          *ya = y;
        }
      }
      if (p.kpos == nullptr) rope_cs8_advance(kcs[n], kstep[n]);
    }
    __syncthreads();
    // ---- scores (log2 units): thread = key kr, rows rg, rg + 4, ... --------------------------
    {
      const int kr = tid % kChunk, rg = tid / kChunk;
      const int j = kc + kr;
      const T* krow = sK + kr * C::KSTRIDE;
      for (int row = rg; row < rows; row += kThreads / kChunk) {
        const int i = row % p.N;
        const float* qrow = sQ + row * D;
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 4
        for (int e = 0; e < D; e += 8) {
          const uint4 kv = *reinterpret_cast<const uint4*>(krow + e);
          const float4 qa = *reinterpret_cast<const float4*>(qrow + e);
          const float4 qb = *reinterpret_cast<const float4*>(qrow + e + 4);
          float k0, k1, k2, k3, k4, k5, k6, k7;
          Pack<BF16>::unpack(kv.x, k0, k1);
          Pack<BF16>::unpack(kv.y, k2, k3);
          Pack<BF16>::unpack(kv.z, k4, k5);
          Pack<BF16>::unpack(kv.w, k6, k7);
          acc0 = fmaf(qa.x, k0, fmaf(qa.y, k1, fmaf(qa.z, k2, fmaf(qa.w, k3, acc0))));
          acc1 = fmaf(qb.x, k4, fmaf(qb.y, k5, fmaf(qb.z, k6, fmaf(qb.w, k7, acc1))));
        }
        const bool visible = j < key_end && j <= p.q_off + i;
        sS[row * kChunk + kr] = visible ? (acc0 + acc1) * p.scale_log2 : -INFINITY;
      }
    }
    __syncthreads();
    // ---- online softmax per row: warp w takes rows w, w + 8, ... -----------------------------
    {
      const int warp = tid / 32, lane = tid % 32;
      for (int row = warp; row < rows; row += kThreads / 32) {
        const float s0 = sS[row * kChunk + lane], s1 = sS[row * kChunk + lane + 32];
        float mx = fmaxf(s0, s1);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
        const float m_old = sM[row];
        const float m_new = fmaxf(m_old, mx);
        // a row that has seen no visible key yet keeps m = -inf, P = 0
        const float p0 = m_new == -INFINITY ? 0.f : ptx::ex2_approx(s0 - m_new);
        const float p1 = m_new == -INFINITY ? 0.f : ptx::ex2_approx(s1 - m_new);
        float sum = p0 + p1;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
        sS[row * kChunk + lane] = p0;
        sS[row * kChunk + lane + 32] = p1;
        __syncwarp();
        if (lane == 0) {
          const float alpha = m_old == -INFINITY ? 0.f : ptx::ex2_approx(m_old - m_new);
          sA[row] = alpha;
          sL[row] = sL[row] * alpha + sum;
          sM[row] = m_new;
        }
      }
    }
    __syncthreads();
    // ---- O = O alpha + P V: thread items (row, column pair) --------------------------------
#pragma unroll
    for (int n = 0; n < kMaxItems; ++n) {
      const int it = tid + kThreads * n;
      if (it >= n_items) break;
      const int row = it / (D / 2), e = 2 * (it % (D / 2));
      const float alpha = sA[row];
      float a0 = oacc[n][0] * alpha, a1 = oacc[n][1] * alpha;
      const float* prow = sS + row * kChunk;
#pragma unroll 8
      for (int kr = 0; kr < kChunk; ++kr) {
        float v0, v1;
        Pack<BF16>::unpack(*reinterpret_cast<const uint32_t*>(sV + kr * D + e), v0, v1);
        const float pw = prow[kr];
        a0 = fmaf(pw, v0, a0);
        a1 = fmaf(pw, v1, a1);
      }
      oacc[n][0] = a0;
      oacc[n][1] = a1;
    }
  }
  // ---- partials of this split ------------------------------------------------------------------
  const size_t base = (((size_t)b * p.Hkv + hk) * p.n_splits + split) * kDecodeMaxRows;
#pragma unroll
  for (int n = 0; n < kMaxItems; ++n) {
    const int it = tid + kThreads * n;
    if (it >= n_items) break;
    const int row = it / (D / 2), e = 2 * (it % (D / 2));
    *reinterpret_cast<float2*>(p.part_o + (base + row) * D + e) = make_float2(oacc[n][0], oacc[n][1]);
  }
  __syncthreads();
  if (tid < rows) {
    p.part_ml[(base + tid) * 2] = sM[tid];
    p.part_ml[(base + tid) * 2 + 1] = sL[tid];
  }
}

// One warp per (batch, KV head, row): m = max_s m_s, l = sum_s l_s 2^(m_s - m),
// out = sum_s O_s 2^(m_s - m) / l, lse = ln 2 (m + log2 l).
template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_decode_combine_kernel(const __grid_constant__ DecodeParams p) {
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  const int g = p.Hq / p.Hkv, rows = g * p.N;
  const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (w >= (long long)p.B * p.Hkv * rows) return;
  const int row = (int)(w % rows);
  const int hk = (int)((w / rows) % p.Hkv);
  const int b = (int)(w / ((long long)rows * p.Hkv));
  const int hl = row / p.N, i = row % p.N, h = hk * g + hl;
  const size_t base = ((size_t)b * p.Hkv + hk) * p.n_splits * kDecodeMaxRows + row;
  float m = -INFINITY;
  for (int s = 0; s < p.n_splits; ++s) m = fmaxf(m, p.part_ml[(base + (size_t)s * kDecodeMaxRows) * 2]);
  constexpr int PER = D / 32;  // columns per lane
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float l = 0.f;
  for (int s = 0; s < p.n_splits; ++s) {
    const size_t slot = base + (size_t)s * kDecodeMaxRows;
    const float ms = p.part_ml[slot * 2];
    if (ms == -INFINITY) continue;  // no visible key of this row in split s
    const float wgt = ptx::ex2_approx(ms - m);
    l = fmaf(p.part_ml[slot * 2 + 1], wgt, l);
    const float* o = p.part_o + slot * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = fmaf(o[e], wgt, acc[e]);
  }
  const float inv = 1.f / l;
  T* dst = reinterpret_cast<T*>(p.out) + (((size_t)b * p.N + i) * p.Hq + h) * D + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; e += 2) {
    const uint32_t wv = Pack<BF16>::pack(acc[e] * inv, acc[e + 1] * inv);
    *reinterpret_cast<uint32_t*>(dst + e) = wv;
  }
  if (lane == 0 && p.lse != nullptr) p.lse[((size_t)b * p.Hq + h) * p.N + i] = (m + log2f(l)) * kLn2;
}

template <int D, bool BF16>
cudaError_t launch_decode_impl(const DecodeParams& p, cudaStream_t stream) {
  constexpr int kMaxDevices = 64;
  static int configured[kMaxDevices] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(attn_decode_kernel<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)DecCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  attn_decode_kernel<D, BF16><<<dim3((unsigned)p.n_splits, (unsigned)p.Hkv, (unsigned)p.B), dim3(kThreads),
                                DecCfg<D>::SMEM, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long warps = (long long)p.B * p.Hkv * (p.Hq / p.Hkv) * p.N;
  const long long blocks = (warps * 32 + 255) / 256;
  attn_decode_combine_kernel<D, BF16><<<dim3((unsigned)blocks), dim3(256), 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_decode(const DecodeParams& p, int d, bool bf16, cudaStream_t stream) {
  if (d == 128) return bf16 ? launch_decode_impl<128, true>(p, stream) : launch_decode_impl<128, false>(p, stream);
  return bf16 ? launch_decode_impl<64, true>(p, stream) : launch_decode_impl<64, false>(p, stream);
}

}  // namespace attnfuse
