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
// attn_decode_kernel: one CTA per (KV head, slice of keys_per_split keys, batch), W warps (eight, or
// twelve in one form, decode_warps) that never wait on one another inside the key loop.  The slice
// is cut into 16-key chunks; warp w takes chunks w, w + W, w + 2 W, ... and owns a ring of
// shared-memory stages (three, or two with twelve warps), each holding one chunk's K and V rows,
// filled by TMA (cp.async.bulk.tensor, 128-byte swizzle) on the warp's own mbarriers, so the warp's
// next chunks are in flight while it computes.  Per chunk the warp rotates the chunk's K rows in
// place (cos/sin carried along the warp's rows and chunks by angle addition, exact again every 16
// chunks; exact per key with explicit positions; rounded to the input type like the other paths),
// computes S = Q K^T for the <= 16 query rows as m16n8k16 tensor-core tiles (Q fragments kept in
// registers), runs the online softmax on the fragments in registers (exp2, fp32 max and sum), and
// adds P V with P passed straight from the score fragments to the operand fragments (P rounded to
// the input type).  At the end the warps' partial (O, max, sum) are merged in shared memory and the
// CTA writes the slice's partial.  One CTA per SM at d = 128 (192 KB of rings), two at d = 64.
// attn_decode_combine_kernel: one CTA per (row, KV head, batch) merges the slices (rescaling each by
// 2^(m_s - m)) into out and lse; launched as a programmatic dependent of the first kernel, it waits
// (griddepcontrol.wait) for that grid to complete before reading the partials.
// Every mbarrier wait is bounded (1 s): a warp that gives up records bit 0 in the decode status word
// (attnfuse_device_status), stops, and lets its copies in flight land before the CTA exits.
#include <cuda_runtime.h>
#include <math.h>

#include <type_traits>

#include "attnfuse_internal.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace attnfuse {

__device__ unsigned int g_decode_status = 0;

namespace {

constexpr int kChunk = kDecodeChunk;  // keys per chunk (one TMA box of rows)
constexpr int kTiles = kChunk / 8;    // 8-key score tiles per chunk
constexpr int kKSteps = kChunk / 16;  // 16-key steps of P V per chunk
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned long long kWaitNs = 1000000000ull;

template <int D, int kWarps, int kStagesPerWarp>
struct DecCfg {
  static constexpr uint32_t BOX = kChunk * 128;                 // kChunk rows x 64 16-bit columns, swizzled
  static constexpr uint32_t KBYTES = (D / 64) * BOX;            // one chunk of K (or V)
  static constexpr uint32_t STAGE = 2 * KBYTES;                 // K then V
  static constexpr int QSTRIDE = D + 8;                         // 16-bit Q rows, padded for ldmatrix
  static constexpr int GPR = D / 16;                            // rotation groups (8 frequencies) per row
  static constexpr int RS = 32 / GPR;                           // rows a warp rotates per pass
  static constexpr int PASSES = kChunk / RS;
  static constexpr uint32_t OFF_RING = 0;
  static constexpr uint32_t OFF_QF = OFF_RING + kWarps * kStagesPerWarp * STAGE;  // fp32 [16][D]
  static constexpr uint32_t OFF_QH = OFF_QF + kDecodeMaxRows * D * 4;             // 16-bit [16][QSTRIDE]
  static constexpr uint32_t OFF_FREQ = OFF_QH + kDecodeMaxRows * QSTRIDE * 2;     // u32 lo[64], hi[64]
  static constexpr uint32_t OFF_STEP = OFF_FREQ + 2 * 64 * 4;                     // RopeCS8 [GPR]: RS rows
  static constexpr uint32_t OFF_SKIP = OFF_STEP + GPR * sizeof(RopeCS8);          // RopeCS8 [GPR]: next chunk
  static constexpr uint32_t OFF_BAR = OFF_SKIP + GPR * sizeof(RopeCS8);           // u64 [warps][stages]
  static constexpr uint32_t SMEM = OFF_BAR + kWarps * kStagesPerWarp * 8 + 1024;  // + alignment slack
  // The warps' partials are merged in the ring after the key loop: O [warps][16][D] and m, l.
  static_assert(kWarps * kDecodeMaxRows * (D + 2) * 4 <= kWarps * kStagesPerWarp * STAGE, "merge area");
  static_assert(OFF_QH % 16 == 0 && OFF_STEP % 16 == 0 && OFF_BAR % 8 == 0, "alignment");
};

// 16-byte chunk `ci` (columns 8 ci .. 8 ci + 7) of row r of a chunk of kChunk rows stored as 128-byte
// swizzled boxes of 64 columns: box ci / 8, logical chunk ci % 8 at physical chunk (ci % 8) ^ (r % 8).
__device__ __forceinline__ uint32_t sw_off(int r, int ci) {
  return (uint32_t)(ci >> 3) * (uint32_t)(kChunk * 128) + (uint32_t)r * 128u + (uint32_t)((((ci & 7) ^ (r & 7))) * 16);
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

// c += a b: a the 16x16 row-major fragment, (b0, b1) the 16x8 column-major fragment (fp32 accumulate).
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

// Bounded wait on a TMA barrier; false (and bit 0 of the decode status word) if it ran out.
__device__ __forceinline__ bool wait_stage(uint32_t bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (;;) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (ptx::globaltimer_ns() - t0 > kWaitNs) {
      atomicOr(&g_decode_status, 1u);
      return false;
    }
  }
}

// R8: at most 8 query rows per KV head (every decode step with groups of up to 8 heads, two tokens of
// groups of four).  The products then use only rows 0..7 of the 16-row tiles, so P V runs
// transposed, O^T = V^T P^T (M = 16 columns of d, N = the 8 rows, K = 16 keys), with P taken
// straight from the score fragments as the B operand; each lane keeps one softmax row.
template <int D, bool BF16, bool R8, int W>
__global__ void __launch_bounds__(32 * W, decode_ctas_per_sm(D))
    attn_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ DecodeParams p) {
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  constexpr int kWarps = W, kThreads = 32 * kWarps, kStagesPerWarp = decode_stages(W);
  using C = DecCfg<D, kWarps, kStagesPerWarp>;
  constexpr int NT = D / 8;    // 8-column output tiles of P V
  constexpr int MT = D / 16;   // R8: 16-column tiles of O^T
  constexpr int KS = D / 16;   // k-steps of Q K^T
  constexpr int NH = R8 ? 1 : 2;  // fragment row halves in use: rows g8 (h = 0) and g8 + 8 (h = 1)
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;  // 128-byte swizzle: 1024-byte aligned boxes
  uint8_t* sgen = smem_raw + (sbase - raw);
  float* sQ = reinterpret_cast<float*>(sgen + C::OFF_QF);
  T* sQh = reinterpret_cast<T*>(sgen + C::OFF_QH);
  uint32_t* sF = reinterpret_cast<uint32_t*>(sgen + C::OFF_FREQ);  // lo[64] then hi[64]
  RopeCS8* sStep = reinterpret_cast<RopeCS8*>(sgen + C::OFF_STEP);
  RopeCS8* sSkip = reinterpret_cast<RopeCS8*>(sgen + C::OFF_SKIP);
  uint64_t* sBar = reinterpret_cast<uint64_t*>(sgen + C::OFF_BAR);

  const int hk = blockIdx.x, split = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int g8 = lane / 4, t4 = lane % 4;  // MMA fragment row and column pair of this lane
  const int g = p.Hq / p.Hkv;
  const int rows = g * p.N;  // row = local head * N + query index
  const int R = p.rot_chunks;  // rotation groups actually rotated (rotary dimension / 16)
  const bool il = p.interleaved != 0;
  const int key0 = split * p.keys_per_split;
  const int key_end = min(p.Nk, key0 + p.keys_per_split);
  const int nch = (key_end - key0 + kChunk - 1) / kChunk;
  const bool skip_all = *reinterpret_cast<volatile unsigned int*>(&g_decode_status) != 0u;

  if (tid == 0) {
    for (int i = 0; i < kWarps * kStagesPerWarp; ++i) ptx::mbar_init(ptx::smem_u32(sBar + i), 1);
    ptx::fence_barrier_init();
  }
  __syncthreads();
  ptx::grid_dep_launch_dependents();  // the combine kernel may launch; it waits for this grid

  // Each warp's first chunks are requested before anything else happens.
  auto stage_addr = [&](int st) { return sbase + C::OFF_RING + (uint32_t)(warp * kStagesPerWarp + st) * C::STAGE; };
  auto issue = [&](int c, int st) {
    const uint32_t bar = ptx::smem_u32(sBar + warp * kStagesPerWarp + st);
    const uint32_t dst = stage_addr(st);
    ptx::mbar_arrive_expect_tx(bar, C::STAGE);
    const int row0 = key0 + kChunk * c;
#pragma unroll
    for (int bx = 0; bx < D / 64; ++bx) {
      ptx::tma_load_4d(dst + bx * C::BOX, &tmK, bar, 64 * bx, hk, row0, b);
      ptx::tma_load_4d(dst + C::KBYTES + bx * C::BOX, &tmV, bar, 64 * bx, hk, row0, b);
    }
  };
  int issued = 0;  // chunks of this warp requested so far (the warp's chunks are warp + kWarps i)
  if (!skip_all && lane == 0) {
    ptx::tma_prefetch_desc(&tmK);
    ptx::tma_prefetch_desc(&tmV);
  }
  if (!skip_all) {
    for (int st = 0; st < kStagesPerWarp; ++st) {
      const int c = warp + kWarps * st;
      if (c >= nch) break;
      if (lane == 0) issue(c, st);
      ++issued;
    }
  }

  // ---- query rows: fp32 in shared memory, rotated exactly per row, rounded once, 16-bit copy ------
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
  if (tid < 64) sF[tid] = p.freqs.lo[tid];
  else if (tid < 128) sF[tid] = p.freqs.hi[tid - 64];
  __syncthreads();
  const int r = 2 * R * 8;  // rotary dimension
  // one rotation pair per thread: row, frequency k = 8 fg + t
  for (int idx = tid; idx < rows * R * 8; idx += kThreads) {
    const int row = idx / (8 * R), kf = idx % (8 * R), fg = kf / 8, t = kf % 8;
    const int i = row % p.N;
    const int32_t pos = p.qpos ? p.qpos[(size_t)b * p.N + i] : p.q_off + i;
    float c, s_;
    rope_cs_signed(pos, sF[kf], sF[64 + kf], c, s_);
    const int ia = il ? 16 * fg + 2 * t : kf;
    const int ib = il ? ia + 1 : r / 2 + ia;
    float xr, yr;
    rope_pair(sQ[row * D + ia], sQ[row * D + ib], c, s_, xr, yr);
    float2 rr;
    Pack<BF16>::unpack(Pack<BF16>::pack(xr, yr), rr.x, rr.y);
    sQ[row * D + ia] = rr.x;
    sQ[row * D + ib] = rr.y;
  }
  // cos/sin steps of a rotation group, one frequency per thread: RS rows (between a lane's passes)
  // and kChunk (kWarps - 1) + RS rows (from a lane's last row of one chunk to its first row of the
  // warp's next chunk).  RopeCS8 holds frequency 8 fg + 2 j + e at float 2 j + e of c (and of s).
  if (tid < 16 * R) {
    const int which = tid / (8 * R), kf = tid % (8 * R), fg = kf / 8, t = kf % 8;
    const uint32_t steps = which == 0 ? (uint32_t)C::RS : (uint32_t)(kChunk * (kWarps - 1) + C::RS);
    float c, s_;
    rope_cs(steps, sF[kf], sF[64 + kf], c, s_);
    float* dst = reinterpret_cast<float*>(which == 0 ? &sStep[fg] : &sSkip[fg]);
    dst[t] = c;
    dst[8 + t] = s_;
  }
  __syncthreads();
  for (int idx = tid; idx < kDecodeMaxRows * (D / 2); idx += kThreads) {
    const int row = idx / (D / 2), e = 2 * (idx % (D / 2));
    const uint32_t w = row < rows ? Pack<BF16>::pack(sQ[row * D + e], sQ[row * D + e + 1]) : 0u;
    *reinterpret_cast<uint32_t*>(sQh + row * C::QSTRIDE + e) = w;
  }
  __syncthreads();
  // Q as A fragments, one per k-step (16 columns), for the whole key loop (R8: rows 8..15 are zero)
  uint32_t qa[KS][4];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    ldsm_x4(ptx::smem_u32(sQh + (lane % 16) * C::QSTRIDE + 16 * ks + 8 * (lane / 16)), qa[ks]);
    if constexpr (R8) qa[ks][1] = qa[ks][3] = 0u;
  }

  // Per lane: rows g8 and g8 + 8 of the fragments; last visible key of each (-1: a padding row).
  int lim[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int row = g8 + 8 * h;
    lim[h] = row < rows ? min(key_end - 1, p.q_off + row % p.N) : -1;
  }
  // Chunks whose keys are all at or before this one are visible to every row (padding rows have no
  // output, so what they compute does not matter): they skip the mask.
  const int lim_all = min(key_end - 1, p.q_off);
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  constexpr int NACC = R8 ? MT : NT;
  float o[NACC][4];  // R8: O^T tiles (columns 16 mt + g8 (+8) of rows 2 t4, 2 t4 + 1); else O tiles
#pragma unroll
  for (int nt = 0; nt < NACC; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

  // Key rotation items of this lane: rotation group fg, rows rsub + RS pass of each chunk.
  const int fg = lane % C::GPR, rsub = lane / C::GPR;
  const bool rot_lane = fg < R;
  const int ca = il ? 2 * fg : fg, cb = il ? 2 * fg + 1 : fg + R;
  RopeCS8 kcs, step;
  if (rot_lane) step = sStep[fg];
  bool ok = !skip_all;
  int done = 0;  // chunks of this warp consumed
  for (int c = warp; ok && c < nch; c += kWarps, ++done) {
    const int st = done % kStagesPerWarp;
    if (!(ok = __all_sync(0xFFFFFFFFu, wait_stage(ptx::smem_u32(sBar + warp * kStagesPerWarp + st),
                                                   (uint32_t)((done / kStagesPerWarp) & 1)))))
      break;
    const uint32_t kst = stage_addr(st), vst = kst + C::KBYTES;
    const int j0 = key0 + kChunk * c;
    // ---- rotate this chunk's K rows in place ------------------------------------------------------
    if (rot_lane) {
      if (p.kpos == nullptr && done % 16 == 0)
        rope_cs8_exact((uint32_t)(j0 + rsub), sF, sF + 64, 8 * fg, kcs);
#pragma unroll
      for (int pass = 0; pass < C::PASSES; ++pass) {
        const int row = rsub + C::RS * pass;
        const int j = j0 + row;
        if (p.kpos != nullptr) {
          const int jc = min(j, p.Nk - 1);  // rows past the sequence hold zeros: any angle will do
          rope_cs8_exact_signed(p.kpos[(size_t)b * p.Nk + jc], sF, sF + 64, 8 * fg, kcs);
        }
        const uint32_t xo = sw_off(row, ca), yo = sw_off(row, cb);
        uint4 x = ptx::lds128(kst + xo), y = ptx::lds128(kst + yo);
        if (il) {
          rope_rotate_chunk_il_cs8<BF16>(x, kcs, 0);
          rope_rotate_chunk_il_cs8<BF16>(y, kcs, 1);
        } else {
          rope_rotate_chunk_cs8<BF16>(x, y, kcs);
        }
        ptx::sts128(kst + xo, x);
        ptx::sts128(kst + yo, y);
        if (p.kpos == nullptr) rope_cs8_advance(kcs, pass + 1 < C::PASSES ? step : sSkip[fg]);
      }
    }
    __syncwarp();
    // ---- S = Q K^T (log2 units): kTiles tiles of 8 keys -------------------------------------------
    float sc[kTiles][4];
#pragma unroll
    for (int nt = 0; nt < kTiles; ++nt) {
      sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ks += 2) {
        uint32_t bk[4];  // keys 8 nt .. 8 nt + 7, columns 16 ks .. 16 ks + 31
        const int krow = 8 * nt + (lane % 8);
        ldsm_x4(kst + sw_off(krow, 2 * ks + lane / 8), bk);
        mma_16816<BF16>(sc[nt], qa[ks], bk[0], bk[1]);
        mma_16816<BF16>(sc[nt], qa[ks + 1], bk[2], bk[3]);
      }
    }
    // ---- online softmax on the fragments: rows g8 (h = 0) and g8 + 8 (h = 1) ----------------------
    const bool masked = j0 + kChunk - 1 > lim_all;  // warp-uniform
    uint32_t pa[kKSteps][4];  // P as the A fragments of the 16-key steps of P V (R8: [0], [2] used)
    bool moved = false;       // some row's running max changed (its O needs the rescale)
    float alpha[2];
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      float sv[2 * kTiles];
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < kTiles; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = j0 + 8 * nt + 2 * t4 + e;
          const float v = (!masked || j <= lim[h]) ? sc[nt][2 * h + e] * p.scale_log2 : -INFINITY;
          sv[2 * nt + e] = v;
          mx = fmaxf(mx, v);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
      const float m_new = fmaxf(m_run[h], mx);
      moved |= m_new != m_run[h];
      // a row that has seen no visible key keeps m = -inf, P = 0, O = 0
      alpha[h] = m_run[h] == -INFINITY ? 0.f : ptx::ex2_approx(m_run[h] - m_new);
      float pv[2 * kTiles], sum = 0.f;
#pragma unroll
      for (int e = 0; e < 2 * kTiles; ++e) {
        pv[e] = m_new == -INFINITY ? 0.f : ptx::ex2_approx(sv[e] - m_new);
        sum += pv[e];
      }
      sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
      sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
      l_run[h] = l_run[h] * alpha[h] + sum;
      m_run[h] = m_new;
      // Score tiles 2 kk and 2 kk + 1 (keys 16 kk .. 16 kk + 15) form the A fragment of key step kk:
      // a0 / a1 = tile 2 kk, rows g8 / g8 + 8; a2 / a3 = tile 2 kk + 1, rows g8 / g8 + 8.  (R8: a0 and
      // a2 are also the B fragment of O^T += V^T P^T for row g8.)
#pragma unroll
      for (int kk = 0; kk < kKSteps; ++kk) {
        pa[kk][h] = Pack<BF16>::pack(pv[4 * kk], pv[4 * kk + 1]);
        pa[kk][2 + h] = Pack<BF16>::pack(pv[4 * kk + 2], pv[4 * kk + 3]);
      }
    }
    // rescale O where a running max moved (most chunks after the first few move none)
    if (__any_sync(0xFFFFFFFFu, moved)) {
      if constexpr (R8) {
        // this lane's O^T columns are rows 2 t4 and 2 t4 + 1, whose alpha lanes 8 t4 and 8 t4 + 4 hold
        const float a0 = __shfl_sync(0xFFFFFFFFu, alpha[0], 8 * t4);
        const float a1 = __shfl_sync(0xFFFFFFFFu, alpha[0], 8 * t4 + 4);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          o[mt][0] *= a0;
          o[mt][1] *= a1;
          o[mt][2] *= a0;
          o[mt][3] *= a1;
        }
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            o[nt][2 * h] *= alpha[h];
            o[nt][2 * h + 1] *= alpha[h];
          }
      }
    }
    if constexpr (R8) {
      // ---- O^T += V^T P^T: per 16 columns of d one ldmatrix (transposed) of V and one MMA ---------
#pragma unroll
      for (int kk = 0; kk < kKSteps; ++kk) {
        // matrices: keys 16 kk + 0..7 / + 8..15 (lane / 16) x columns 16 mt + 0..7 / + 8..15 ((lane / 8) % 2)
        const int vrow = 16 * kk + (lane % 8) + 8 * (lane / 16);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t av[4];
          ldsm_x4_trans(vst + sw_off(vrow, 2 * mt + (lane / 8) % 2), av);
          mma_16816<BF16>(o[mt], av, pa[kk][0], pa[kk][2]);
        }
      }
    } else {
      // ---- O += P V: 16 keys per step, 16 columns per ldmatrix ----------------------------------
#pragma unroll
      for (int kk = 0; kk < kKSteps; ++kk) {
        const int vrow = 16 * kk + (lane % 8) + 8 * ((lane / 8) % 2);
#pragma unroll
        for (int n2 = 0; n2 < NT / 2; ++n2) {
          uint32_t bv[4];  // keys 16 kk .. +15, columns 16 n2 .. +7 (bv[0..1]) and +8 .. +15 (bv[2..3])
          ldsm_x4_trans(vst + sw_off(vrow, 2 * n2 + lane / 16), bv);
          mma_16816<BF16>(o[2 * n2], pa[kk], bv[0], bv[1]);
          mma_16816<BF16>(o[2 * n2 + 1], pa[kk], bv[2], bv[3]);
        }
      }
    }
    __syncwarp();
    // ---- refill this stage with the warp's chunk kStagesPerWarp steps ahead ------------------------
    const int cn = c + kWarps * kStagesPerWarp;
    if (cn < nch) {
      if (lane == 0) {
        ptx::fence_proxy_async_smem();  // this warp's reads of the stage before TMA overwrites it
        issue(cn, st);
      }
      ++issued;
    }
  }
  // Copies still in flight (only after a wait ran out) must land before shared memory is released.
  if (lane == 0)
    for (int k = done; k < issued; ++k) {
      const uint32_t bar = ptx::smem_u32(sBar + warp * kStagesPerWarp + k % kStagesPerWarp);
      const uint64_t t0 = ptx::globaltimer_ns();
      while (!ptx::mbar_try_wait(bar, (uint32_t)((k / kStagesPerWarp) & 1)))
        if (ptx::globaltimer_ns() - t0 > kWaitNs) break;
    }
  __syncthreads();

  // ---- merge the warps' partials in the ring, write this slice's (O, m, l) ----------------------
  float* mO = reinterpret_cast<float*>(sgen + C::OFF_RING);     // [warps][16][D]
  float* mM = mO + kWarps * kDecodeMaxRows * D;                 // [warps][16]
  float* mL = mM + kWarps * kDecodeMaxRows;                     // [warps][16]
  if constexpr (R8) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = 2 * t4 + (e & 1), col = 16 * mt + g8 + 8 * (e >> 1);
        mO[(warp * kDecodeMaxRows + row) * D + col] = o[mt][e];
      }
  } else {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = g8 + 8 * h, col = 8 * nt + 2 * t4;
        *reinterpret_cast<float2*>(mO + (warp * kDecodeMaxRows + row) * D + col) =
            make_float2(o[nt][2 * h], o[nt][2 * h + 1]);
      }
  }
  if (t4 == 0)
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      mM[warp * kDecodeMaxRows + g8 + 8 * h] = m_run[h];
      mL[warp * kDecodeMaxRows + g8 + 8 * h] = l_run[h];
    }
  __syncthreads();
  const size_t base = (((size_t)b * p.Hkv + hk) * p.n_splits + split) * kDecodeMaxRows;
  for (int idx = tid; idx < rows * D; idx += kThreads) {
    const int row = idx / D, col = idx % D;
    float m = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) m = fmaxf(m, mM[w * kDecodeMaxRows + row]);
    float acc = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = mM[w * kDecodeMaxRows + row];
      const float wt = mw == -INFINITY ? 0.f : ptx::ex2_approx(mw - m);
      acc = fmaf(mO[(w * kDecodeMaxRows + row) * D + col], wt, acc);
      l = fmaf(mL[w * kDecodeMaxRows + row], wt, l);
    }
    p.part_o[(base + row) * D + col] = acc;
    if (col == 0) {
      p.part_ml[(base + row) * 2] = m;
      p.part_ml[(base + row) * 2 + 1] = l;
    }
  }
}

// One CTA of 128 threads per (row, KV head, batch): m = max_s m_s, w_s = 2^(m_s - m),
// l = sum_s l_s w_s, out = sum_s O_s w_s / l, lse = ln 2 (m + log2 l).  Warp w takes splits w,
// w + 4, w + 8, ... in batches of kBatch: every load of a batch -- each split's (m, l) pair and the
// lane's 4 (or 2) columns of its O row -- is issued before any is used, so up to 4 kBatch = 32
// splits cost one round of loads; the warp merges its batches online (running max, rescaled sums),
// and a shared-memory pass merges the 4 warps.  A split with no visible key of this row has m =
// -inf (weight 0).
// 128 threads: beside an eight-warp decode CTA (at most 228 registers x 256 threads) a combine CTA
// still fits (registers and shared memory), so the programmatic dependent's CTAs are resident and
// waiting when the decode grid finishes; beside the twelve-warp form they take the SMs it leaves.
constexpr int kCombineThreads = 128;
constexpr int kMaxSplits = 1024;  // decode_plan never makes more
constexpr int kBatch = 8;         // splits per warp whose loads are in flight together

template <int D, bool BF16>
__global__ void __launch_bounds__(kCombineThreads) attn_decode_combine_kernel(const __grid_constant__ DecodeParams p) {
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  constexpr int NW = kCombineThreads / 32;
  constexpr int PER = D / 32;  // columns per lane
  __shared__ float s_acc[NW][D];
  __shared__ float s_ml[NW][2];
  const int row = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int g = p.Hq / p.Hkv;
  const int hl = row / p.N, i = row % p.N, h = hk * g + hl;
  const size_t base = ((size_t)b * p.Hkv + hk) * p.n_splits * kDecodeMaxRows + row;
  const int S = p.n_splits;
  ptx::grid_dep_wait();  // the partials of every split are complete and visible
  float m_w = -INFINITY, l_w = 0.f, acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  for (int s0 = warp; s0 < S; s0 += NW * kBatch) {
    float ms[kBatch], ls[kBatch], os[kBatch][PER];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int sp = s0 + NW * k;
      ms[k] = -INFINITY;
      ls[k] = 0.f;
#pragma unroll
      for (int e = 0; e < PER; ++e) os[k][e] = 0.f;
      if (sp < S) {
        const size_t slot = base + (size_t)sp * kDecodeMaxRows;
        const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + slot * 2);
        ms[k] = ml.x;
        ls[k] = ml.y;
        const float* o = p.part_o + slot * D + lane * PER;
        if constexpr (PER == 4) {
          const float4 v = *reinterpret_cast<const float4*>(o);
          os[k][0] = v.x;
          os[k][1] = v.y;
          os[k][2] = v.z;
          os[k][3] = v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2*>(o);
          os[k][0] = v.x;
          os[k][1] = v.y;
        }
      }
    }
    float mb = m_w;
#pragma unroll
    for (int k = 0; k < kBatch; ++k) mb = fmaxf(mb, ms[k]);
    if (mb == -INFINITY) continue;  // nothing visible so far
    const float r = m_w == -INFINITY ? 0.f : ptx::ex2_approx(m_w - mb);
    l_w *= r;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] *= r;
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const float wk = ms[k] == -INFINITY ? 0.f : ptx::ex2_approx(ms[k] - mb);
      l_w = fmaf(ls[k], wk, l_w);
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] = fmaf(os[k][e], wk, acc[e]);
    }
    m_w = mb;
  }
#pragma unroll
  for (int e = 0; e < PER; ++e) s_acc[warp][lane * PER + e] = acc[e];
  if (lane == 0) {
    s_ml[warp][0] = m_w;
    s_ml[warp][1] = l_w;
  }
  __syncthreads();
  if (tid < D / 2) {
    float m = s_ml[0][0];
#pragma unroll
    for (int k = 1; k < NW; ++k) m = fmaxf(m, s_ml[k][0]);
    float l = 0.f, x0 = 0.f, x1 = 0.f;
#pragma unroll
    for (int k = 0; k < NW; ++k) {
      const float wk = s_ml[k][0] == -INFINITY ? 0.f : ptx::ex2_approx(s_ml[k][0] - m);
      l = fmaf(s_ml[k][1], wk, l);
      x0 = fmaf(s_acc[k][2 * tid], wk, x0);
      x1 = fmaf(s_acc[k][2 * tid + 1], wk, x1);
    }
    const float inv = 1.f / l;
    T* dst = reinterpret_cast<T*>(p.out) + (((size_t)b * p.N + i) * p.Hq + h) * D + 2 * tid;
    *reinterpret_cast<uint32_t*>(dst) = Pack<BF16>::pack(x0 * inv, x1 * inv);
    if (tid == 0 && p.lse != nullptr) p.lse[((size_t)b * p.Hq + h) * p.N + i] = (m + log2f(l)) * kLn2;
  }
}

template <int D, bool BF16, bool R8, int W>
cudaError_t launch_decode_kernel(const DecodeMaps& maps, const DecodeParams& p, cudaStream_t stream) {
  using Cfg = DecCfg<D, W, decode_stages(W)>;
  static DeviceOnce once;  // shared-memory attribute set once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int unused = 0;
  e = once.get(dev, [](int*) -> cudaError_t {
    return cudaFuncSetAttribute(attn_decode_kernel<D, BF16, R8, W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)Cfg::SMEM);
  }, &unused);
  if (e != cudaSuccess) return e;
  attn_decode_kernel<D, BF16, R8, W><<<dim3((unsigned)p.Hkv, (unsigned)p.n_splits, (unsigned)p.B), dim3(32 * W),
                                       Cfg::SMEM, stream>>>(maps.k, maps.v, p);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_decode_impl(const DecodeMaps& maps, const DecodeParams& p, cudaStream_t stream) {
  const int rows = (p.Hq / p.Hkv) * p.N;
  cudaError_t e;
  if (rows > 8) {
    e = launch_decode_kernel<D, BF16, false, 8>(maps, p, stream);
  } else if constexpr (D == 128) {
    e = p.warps == 12 ? launch_decode_kernel<D, BF16, true, 12>(maps, p, stream)
                      : launch_decode_kernel<D, BF16, true, 8>(maps, p, stream);
  } else {
    e = launch_decode_kernel<D, BF16, true, 8>(maps, p, stream);
  }
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

cudaError_t launch_attn_decode(const DecodeMaps& maps, const DecodeParams& p, int d, bool bf16, cudaStream_t stream) {
  if (d == 128)
    return bf16 ? launch_decode_impl<128, true>(maps, p, stream) : launch_decode_impl<128, false>(maps, p, stream);
  return bf16 ? launch_decode_impl<64, true>(maps, p, stream) : launch_decode_impl<64, false>(maps, p, stream);
}

cudaError_t read_and_clear_decode_status(unsigned int* value) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_decode_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  if (*value != 0u) {
    const unsigned int zero = 0u;
    e = cudaMemcpyToSymbol(g_decode_status, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace attnfuse
