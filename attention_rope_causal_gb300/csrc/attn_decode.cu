// Causal RoPE attention for a few queries against many keys (decode, speculative decode): split-KV.
// With N queries and rows = (Hq / Hkv) N <= 16 query rows per KV head the 128-row tile kernels keep
// at most one useful row in eight and walk each KV head's keys in one CTA; here the keys of every
// KV head are split over many CTAs and the products run as 16-row tensor-core tiles.
//
// What it computes: the function of attnfuse_rope_causal_fwd (header of include/attnfuse.h) in
// its general form -- the N queries are the last N of the Nk tokens, query i sees keys j <= Nk - N
// + i, rotation positions q_off + i and j or the explicit arrays, any rotary dimension and pairing
// ("AttnFuse Makes RoPE a First-Class Attention Compilation Operation", paragraphs 1-2: RoPE on Q
// and K before the product, causal mask, softmax).
//
// attn_decode_kernel: one CTA per (KV head, split of keys_per_split keys, batch), 256 threads, two
// (d = 128) or three (d = 64) CTAs per SM.  The CTA rotates its query rows once (exact cos/sin per row) into fp32 shared
// memory, then walks its keys 64 at a time: the next chunk's K and V rows are loaded into registers
// (16-byte loads) while the current chunk is processed; K is rotated in shared memory by cos/sin
// carried from chunk to chunk (advanced by the exact rotation of 64 positions, recomputed exactly
// every 16 chunks; exact per key with explicit positions) and rounded to the input type like the
// other paths; S = Q K^T by m16n8k16 MMAs (warp w: keys 8w .. 8w + 7), online softmax per row (exp2,
// fp32 max and sum, P rounded to the input type), O += P V by MMAs (warp w: 8 d / 64 columns) with
// the accumulators in registers.  It writes the unnormalised O, the running max (log2 units) and the
// sum of its split.
// attn_decode_combine_kernel: one CTA per (row, KV head, batch) merges the splits (rescaling each by
// 2^(m_s - m)) into out and lse; launched as a programmatic dependent of the first kernel, it waits
// (griddepcontrol.wait) for that grid to complete before reading the partials.
// No spin-waits: the first kernel synchronises only with __syncthreads, so the second one's wait
// ends when the first grid does.
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
  // 16-bit elements per row of the Q, K and V tiles in shared memory: consecutive rows 16 bytes apart
  // modulo 128, so the eight row addresses of an ldmatrix fall in distinct banks.
  static constexpr int KSTRIDE = D + 8;
  static constexpr int PSTRIDE = kChunk + 8;  // the same for P
  static constexpr uint32_t OFF_Q = 0;                                          // fp32 [16][D]
  static constexpr uint32_t OFF_QH = OFF_Q + kDecodeMaxRows * D * 4;            // 16-bit [16][KSTRIDE]
  static constexpr uint32_t OFF_K = OFF_QH + kDecodeMaxRows * KSTRIDE * 2;      // 16-bit [64][KSTRIDE]
  static constexpr uint32_t OFF_V = OFF_K + kChunk * KSTRIDE * 2;               // 16-bit [64][KSTRIDE]
  static constexpr int SSTRIDE = kChunk + 8;  // fp32 scores per row: the eight rows of an MMA
                                              // fragment's store fall in distinct banks
  static constexpr uint32_t OFF_S = OFF_V + kChunk * KSTRIDE * 2;               // fp32 [16][SSTRIDE]
  static constexpr uint32_t OFF_P = OFF_S + kDecodeMaxRows * SSTRIDE * 4;       // 16-bit [16][PSTRIDE]
  static constexpr uint32_t OFF_ROW = OFF_P + kDecodeMaxRows * PSTRIDE * 2;     // fp32 [16] m, l, alpha
  static constexpr uint32_t OFF_FREQ = OFF_ROW + 3 * kDecodeMaxRows * 4;        // u32 F_k lo[64], hi[64]
  static constexpr uint32_t OFF_STEP = OFF_FREQ + 2 * 64 * 4;                   // u64 c[4][8], s[4][8]
  static constexpr uint32_t SMEM = OFF_STEP + 8 * sizeof(RopeCS8);
  static_assert(OFF_QH % 16 == 0 && OFF_K % 16 == 0 && OFF_V % 16 == 0 && OFF_P % 16 == 0 && OFF_STEP % 16 == 0,
                "ldmatrix rows and 16-byte stores need 16-byte aligned regions");
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

// Warp-level tensor-core products for the (<= 16)-row tiles: ldmatrix fragments and the
// m16n8k16 MMA (fp32 accumulators).  tcgen05's smallest M (64) would leave three quarters of
// every product empty here.
__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x2_trans(uint32_t addr, uint32_t (&r)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr)
               : "memory");
}

// c += a b: a the 16x16 row-major fragment, (b0, b1) the 16x8 column-major fragment.
template <bool BF16>
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, decode_ctas_per_sm(D)) attn_decode_kernel(const __grid_constant__ DecodeParams p) {
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  using C = DecCfg<D>;
  constexpr int KS = C::KSTRIDE;
  constexpr int NT = D / 64;  // 8-column output tiles per warp in P V (8 warps cover d columns)
  extern __shared__ __align__(16) uint8_t smem[];
  float* sQ = reinterpret_cast<float*>(smem + C::OFF_Q);
  T* sQh = reinterpret_cast<T*>(smem + C::OFF_QH);
  T* sK = reinterpret_cast<T*>(smem + C::OFF_K);
  T* sV = reinterpret_cast<T*>(smem + C::OFF_V);
  float* sS = reinterpret_cast<float*>(smem + C::OFF_S);
  T* sP = reinterpret_cast<T*>(smem + C::OFF_P);
  float* sM = reinterpret_cast<float*>(smem + C::OFF_ROW);
  float* sL = sM + kDecodeMaxRows;
  float* sA = sL + kDecodeMaxRows;
  uint32_t* sF = reinterpret_cast<uint32_t*>(smem + C::OFF_FREQ);  // lo[64] then hi[64]
  // cos/sin of 64 positions per frequency group, field-major ([j][group]) so that the lanes of a
  // warp, which hold consecutive groups, read consecutive words
  uint64_t* sStepC = reinterpret_cast<uint64_t*>(smem + C::OFF_STEP);
  uint64_t* sStepS = sStepC + 4 * 8;

  // KV head fastest: CTAs launched together read the same key rows of all heads (whole DRAM pages)
  const int hk = blockIdx.x, split = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int g8 = lane / 4, t4 = lane % 4;  // MMA fragment row and column-pair of this lane
  // the combine kernel may launch now; it waits for this grid's completion before reading
  ptx::grid_dep_launch_dependents();
  const int g = p.Hq / p.Hkv;
  const int rows = g * p.N;  // row = local head * N + query index
  const int r = 2 * p.rot_chunks * 8;  // rotary dimension
  const bool il = p.interleaved != 0;
  const int key0 = split * p.keys_per_split;
  const int key_end = min(p.Nk, key0 + p.keys_per_split);

  // K and V rows of a chunk: warp w loads rows 8w .. 8w + 7 (LPT 16-byte pieces per lane, 16 or 8
  // lanes per row), all loads issued before any is used; the next chunk's are in flight while the
  // current one is computed on, the first chunk's while the query rows are prepared.
  constexpr int LPT = D / 32;  // 4 (d = 128) or 2 (d = 64)
  uint4 kpre[LPT], vpre[LPT];
  auto piece = [&](int n, int& kr, int& c8) {
    const int local = 32 * n + lane;
    kr = 8 * warp + local / (D / 8);
    c8 = local % (D / 8);
  };
  auto load_chunk = [&](int kc) {
#pragma unroll
    for (int n = 0; n < LPT; ++n) {
      int kr, c8;
      piece(n, kr, c8);
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

  // ---- query rows into fp32 shared memory; row state; P's padding rows stay zero ----------------
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
    sA[tid] = 0.f;
  }
  for (int idx = tid; idx < kDecodeMaxRows * C::PSTRIDE / 2; idx += kThreads) reinterpret_cast<uint32_t*>(sP)[idx] = 0u;
  // F_k in shared memory: per-lane frequency indices would serialise constant-bank loads.
  if (tid < 64) sF[tid] = p.freqs.lo[tid];
  else if (tid < 128) sF[tid] = p.freqs.hi[tid - 64];
  __syncthreads();
  // ---- rotate the query rows (exact cos/sin per row), rounded to the input type once --------------
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
      float2 rr;
      Pack<BF16>::unpack(Pack<BF16>::pack(xr, yr), rr.x, rr.y);
      sQ[row * D + ia] = rr.x;
      sQ[row * D + ib] = rr.y;
    }
  }
  if (tid < p.rot_chunks) {
    RopeCS8 st;
    rope_cs8_exact((uint32_t)kChunk, sF, sF + 64, 8 * tid, st);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      sStepC[8 * j + tid] = st.c[j];
      sStepS[8 * j + tid] = st.s[j];
    }
  }
  __syncthreads();
  // 16-bit copy for the MMA (exact: every entry is a value of the input type); rows >= rows zero.
  for (int idx = tid; idx < kDecodeMaxRows * (D / 2); idx += kThreads) {
    const int row = idx / (D / 2), e = 2 * (idx % (D / 2));
    const uint32_t w = row < rows ? Pack<BF16>::pack(sQ[row * D + e], sQ[row * D + e + 1]) : 0u;
    *reinterpret_cast<uint32_t*>(sQh + row * KS + e) = w;
  }
  // (read by every warp as A fragments in each chunk's score product: sQh is stable from here on)

  // O accumulators of this warp: rows g8 and g8 + 8, columns n0 + 8 nt + 2 t4 (+1).
  const int n0 = warp * 8 * NT;
  float o[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

  // cos/sin of the thread's key-rotation items (see below); their advance by 64 positions is shared
  // per frequency group (sStepC, sStepS).
  constexpr int KIT = D / 64;  // rotation items per lane: 8 keys x at most D/16 groups per warp
  RopeCS8 kcs[KIT];

  for (int kc = key0; kc < key_end; kc += kChunk) {
    __syncthreads();  // every warp is done with the previous chunk's V and P
    // Warp w owns K rows 8w .. 8w + 7 from the store through the rotation to the score product, so
    // only V (read by every warp) needs the CTA-wide barriers.
#pragma unroll
    for (int n = 0; n < LPT; ++n) {
      int kr, c8;
      piece(n, kr, c8);
      *reinterpret_cast<uint4*>(sK + kr * KS + 8 * c8) = kpre[n];
      *reinterpret_cast<uint4*>(sV + kr * KS + 8 * c8) = vpre[n];
    }
    if (kc + kChunk < key_end) load_chunk(kc + kChunk);
    __syncwarp();
    // ---- rotate the warp's keys in place -------------------------------------------------------
    // Lane item n: key row kr, frequency group fg (8 frequencies, two 16-byte pieces).  Positions
    // j: cos/sin carried from chunk to chunk by the exact rotation of 64 positions, exact again every
    // 16 chunks; explicit positions: exact per key.
#pragma unroll
    for (int n = 0; n < KIT; ++n) {
      const int local = 32 * n + lane;
      if (local >= 8 * p.rot_chunks) break;
      const int kr = 8 * warp + local / p.rot_chunks, fg = local % p.rot_chunks;
      const int j = kc + kr;
      if (p.kpos != nullptr) {
        if (j < key_end) rope_cs8_exact_signed(p.kpos[(size_t)b * p.Nk + j], sF, sF + 64, 8 * fg, kcs[n]);
      } else if (((kc - key0) / kChunk) % 16 == 0) {
        rope_cs8_exact((uint32_t)j, sF, sF + 64, 8 * fg, kcs[n]);
      }
      if (j < key_end) {
        T* row = sK + kr * KS;
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
      if (p.kpos == nullptr) {
        RopeCS8 st;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          st.c[jj] = sStepC[8 * jj + fg];
          st.s[jj] = sStepS[8 * jj + fg];
        }
        rope_cs8_advance(kcs[n], st);
      }
    }
    __syncwarp();
    // ---- scores (log2 units) S = Q K^T: warp w takes keys 8w .. 8w + 7 -------------------------
    {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < D / 16; ks += 2) {
        uint32_t qa0[4], qa1[4], bk[4];  // query k-steps ks, ks + 1; the keys' 16x8 fragments of both
        ldsm_x4(smem_u32(sQh + (lane % 16) * KS + 16 * ks + 8 * (lane / 16)), qa0);
        ldsm_x4(smem_u32(sQh + (lane % 16) * KS + 16 * (ks + 1) + 8 * (lane / 16)), qa1);
        ldsm_x4(smem_u32(sK + (8 * warp + lane % 8) * KS + 16 * ks + 8 * (lane / 8)), bk);
        mma_16816<BF16>(c, qa0, bk[0], bk[1]);
        mma_16816<BF16>(c, qa1, bk[2], bk[3]);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = g8 + 8 * h;
        if (row < rows) {
          const int i = row % p.N;
          const int kr = 8 * warp + 2 * t4, j = kc + kr;
          const int lim = min(key_end - 1, p.q_off + i);  // last visible key
          *reinterpret_cast<float2*>(sS + row * C::SSTRIDE + kr) =
              make_float2(j <= lim ? c[2 * h] * p.scale_log2 : -INFINITY,
                          j + 1 <= lim ? c[2 * h + 1] * p.scale_log2 : -INFINITY);
        }
      }
    }
    __syncthreads();
    // ---- online softmax per row: warp w takes rows w, w + 8 -----------------------------------
    for (int row = warp; row < rows; row += kThreads / 32) {
      const float s0 = sS[row * C::SSTRIDE + lane], s1 = sS[row * C::SSTRIDE + lane + 32];
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
      // P rounded to the input type for the product, like the tile kernels
      sP[row * C::PSTRIDE + lane] = static_cast<T>(p0);
      sP[row * C::PSTRIDE + lane + 32] = static_cast<T>(p1);
      if (lane == 0) {
        const float alpha = m_old == -INFINITY ? 0.f : ptx::ex2_approx(m_old - m_new);
        sA[row] = alpha;
        sL[row] = sL[row] * alpha + sum;
        sM[row] = m_new;
      }
    }
    __syncthreads();
    // ---- O = O alpha + P V: warp w takes columns n0 .. n0 + 8 NT - 1 ---------------------------
    {
      const float a_lo = sA[g8], a_hi = sA[g8 + 8];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        o[nt][0] *= a_lo;
        o[nt][1] *= a_lo;
        o[nt][2] *= a_hi;
        o[nt][3] *= a_hi;
      }
#pragma unroll
      for (int kk = 0; kk < kChunk / 16; ++kk) {
        uint32_t pa[4];
        ldsm_x4(smem_u32(sP + (lane % 16) * C::PSTRIDE + 16 * kk + 8 * (lane / 16)), pa);
        const int mi = lane / 8;
        if constexpr (NT == 2) {
          uint32_t bv[4];  // keys 16 kk .. +15 of columns n0 .. n0 + 7 and n0 + 8 .. n0 + 15
          ldsm_x4_trans(smem_u32(sV + (16 * kk + lane % 8 + 8 * (mi % 2)) * KS + n0 + 8 * (mi / 2)), bv);
          mma_16816<BF16>(o[0], pa, bv[0], bv[1]);
          mma_16816<BF16>(o[1], pa, bv[2], bv[3]);
        } else {
          uint32_t bv[2];
          ldsm_x2_trans(smem_u32(sV + (16 * kk + lane % 8 + 8 * (mi % 2)) * KS + n0), bv);
          mma_16816<BF16>(o[0], pa, bv[0], bv[1]);
        }
      }
    }
  }
  // ---- partials of this split ------------------------------------------------------------------
  const size_t base = (((size_t)b * p.Hkv + hk) * p.n_splits + split) * kDecodeMaxRows;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = g8 + 8 * h;
      if (row < rows) {
        const int col = n0 + 8 * nt + 2 * t4;
        *reinterpret_cast<float2*>(p.part_o + (base + row) * D + col) = make_float2(o[nt][2 * h], o[nt][2 * h + 1]);
      }
    }
  }
  __syncthreads();
  if (tid < rows) {
    p.part_ml[(base + tid) * 2] = sM[tid];
    p.part_ml[(base + tid) * 2 + 1] = sL[tid];
  }
}

// One CTA of 256 threads per (row, KV head, batch): m = max_s m_s, w_s = 2^(m_s - m),
// l = sum_s l_s w_s, out = sum_s O_s w_s / l, lse = ln 2 (m + log2 l).  The splits' (m, l) pairs
// are read in one pass by as many threads, the weights go to shared memory, and each of the 8 warps
// sums the O rows of every 8th split (lane = 4 or 2 consecutive columns) with loads that do not
// depend on one another; a shared-memory pass adds the 8 warps' sums.  Two rounds of loads in all,
// whatever the number of splits.
constexpr int kCombineThreads = 256;
constexpr int kMaxSplits = 1024;  // decode_plan never makes more

template <int D, bool BF16>
__global__ void __launch_bounds__(kCombineThreads) attn_decode_combine_kernel(const __grid_constant__ DecodeParams p) {
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  constexpr int NW = kCombineThreads / 32;
  constexpr int PER = D / 32;  // columns per lane
  __shared__ float s_w[kMaxSplits];
  __shared__ float s_red[NW][D];
  __shared__ float s_part[2][NW];
  const int row = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int g = p.Hq / p.Hkv;
  const int hl = row / p.N, i = row % p.N, h = hk * g + hl;
  const size_t base = ((size_t)b * p.Hkv + hk) * p.n_splits * kDecodeMaxRows + row;
  const int S = p.n_splits;
  ptx::grid_dep_wait();  // the partials of every split are complete and visible
  // (m, l) of this thread's splits; a split with no visible key of this row has m = -inf (weight 0)
  float m_loc = -INFINITY;
  for (int s = tid; s < S; s += kCombineThreads) {
    const float ms = p.part_ml[(base + (size_t)s * kDecodeMaxRows) * 2];
    s_w[s] = ms;
    m_loc = fmaxf(m_loc, ms);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m_loc = fmaxf(m_loc, __shfl_xor_sync(0xFFFFFFFFu, m_loc, off));
  if (lane == 0) s_part[0][warp] = m_loc;
  __syncthreads();
  float m = s_part[0][0];
#pragma unroll
  for (int k = 1; k < NW; ++k) m = fmaxf(m, s_part[0][k]);
  float l_loc = 0.f;
  for (int s = tid; s < S; s += kCombineThreads) {
    const float ms = s_w[s];
    const float wgt = ms == -INFINITY ? 0.f : ptx::ex2_approx(ms - m);
    s_w[s] = wgt;
    if (wgt != 0.f) l_loc = fmaf(p.part_ml[(base + (size_t)s * kDecodeMaxRows) * 2 + 1], wgt, l_loc);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l_loc += __shfl_xor_sync(0xFFFFFFFFu, l_loc, off);
  if (lane == 0) s_part[1][warp] = l_loc;
  __syncthreads();
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
#pragma unroll 4
  for (int s = warp; s < S; s += NW) {
    const float wu = s_w[s];
    const float* o = p.part_o + (base + (size_t)s * kDecodeMaxRows) * D + lane * PER;
    if constexpr (PER == 4) {
      const float4 v = *reinterpret_cast<const float4*>(o);
      acc[0] = fmaf(v.x, wu, acc[0]);
      acc[1] = fmaf(v.y, wu, acc[1]);
      acc[2] = fmaf(v.z, wu, acc[2]);
      acc[3] = fmaf(v.w, wu, acc[3]);
    } else {
      const float2 v = *reinterpret_cast<const float2*>(o);
      acc[0] = fmaf(v.x, wu, acc[0]);
      acc[1] = fmaf(v.y, wu, acc[1]);
    }
  }
#pragma unroll
  for (int e = 0; e < PER; ++e) s_red[warp][lane * PER + e] = acc[e];
  __syncthreads();
  if (tid < D / 2) {
    float l = 0.f;
#pragma unroll
    for (int k = 0; k < NW; ++k) l += s_part[1][k];
    const float inv = 1.f / l;
    float x0 = 0.f, x1 = 0.f;
#pragma unroll
    for (int k = 0; k < NW; ++k) {
      x0 += s_red[k][2 * tid];
      x1 += s_red[k][2 * tid + 1];
    }
    T* dst = reinterpret_cast<T*>(p.out) + (((size_t)b * p.N + i) * p.Hq + h) * D + 2 * tid;
    *reinterpret_cast<uint32_t*>(dst) = Pack<BF16>::pack(x0 * inv, x1 * inv);
    if (tid == 0 && p.lse != nullptr) p.lse[((size_t)b * p.Hq + h) * p.N + i] = (m + log2f(l)) * kLn2;
  }
}

template <int D, bool BF16>
cudaError_t launch_decode_impl(const DecodeParams& p, cudaStream_t stream) {
  static DeviceOnce once;  // shared-memory attribute set once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int unused = 0;
  e = once.get(dev, [](int*) -> cudaError_t {
    return cudaFuncSetAttribute(attn_decode_kernel<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)DecCfg<D>::SMEM);
  }, &unused);
  if (e != cudaSuccess) return e;
  attn_decode_kernel<D, BF16><<<dim3((unsigned)p.Hkv, (unsigned)p.n_splits, (unsigned)p.B), dim3(kThreads),
                                DecCfg<D>::SMEM, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.n_splits > kMaxSplits) return cudaErrorInvalidConfiguration;
  // Programmatic dependent launch: the combine grid's launch overlaps the decode grid's tail.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((p.Hq / p.Hkv) * p.N), (unsigned)p.Hkv, (unsigned)p.B);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_decode_combine_kernel<D, BF16>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_decode(const DecodeParams& p, int d, bool bf16, cudaStream_t stream) {
  if (d == 128) return bf16 ? launch_decode_impl<128, true>(p, stream) : launch_decode_impl<128, false>(p, stream);
  return bf16 ? launch_decode_impl<64, true>(p, stream) : launch_decode_impl<64, false>(p, stream);
}

}  // namespace attnfuse
