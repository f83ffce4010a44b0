// Backward pass of causal softmax attention with RoPE on sm_103a: dq, dk, dv from q, k, v, the
// forward's output O and log-sum-exp, and dO = dL/dO.
//
// What it computes (the chain rule through the forward of "AttnFuse Makes RoPE a First-Class
// Attention Compilation Operation", 2026-09-13 AI papers report, paragraphs 1-2: RoPE on Q and K
// before the product, causal mask, softmax; training needs this pass, paragraph 3): with q' = R(i) q,
// k' = R(j) k, P_ij = exp(q'_i.k'_j / sqrt(d) - lse_i) for j <= i,
//   dv_j  = sum_{h in the group, i >= j} P_ij dO_i
//   dS_ij = P_ij (dO_i . v_j - D_i),   D_i = dO_i . O_i  (= sum_j P_ij dO_i . v_j)
//   dq_i  = R(i)^T sum_j dS_ij k'_j / sqrt(d),   dk_j = R(j)^T sum_{h, i >= j} dS_ij q'_i / sqrt(d)
// (R^T: the rotation by the negated angle).  Three steps:
//   1. the pre-rotation kernel writes q', k' to the workspace, and bwd_prep_kernel writes D;
//   2. bwd_dkdv_kernel: one unit = one 128-key tile of one KV head; it walks every query tile at or
//      after the key tile, for every query head of the group, accumulating dV and dK' in tensor
//      memory (S^T = K' Q'^T and dP^T = V dO^T by tcgen05.mma, P^T and dS^T elementwise, then
//      dV += P^T dO and dK' += dS^T Q' with P^T, dS^T read from tensor memory);
//   3. bwd_dq_kernel: one unit = one 128-row query tile of one head; it walks key tiles 0 .. its
//      diagonal, accumulating dQ' (S and dP, dS elementwise, dQ' += dS K').
// Both epilogues scale by 1/sqrt(d) and, for the half-split form at positions i and j, rotate back
// with R^T at the row's position in registers (a thread holds a whole row, so each pair (e, e + d/2)
// is local); other RoPE forms and explicit positions leave that to a pre-rotation pass run with the
// negated positions.
//
// Structure of both kernels: 384 threads, one CTA per SM, persistent over units.
//   warp 0      TMA producer (whole warp; lane 0 issues), also stages lse/D vectors for dK/dV.
//   warp 1      tcgen05.mma issuer (whole warp, one elected lane issues); owns the tensor memory.
//   warps 4-7   elementwise for columns 0..63 of each 128 x 128 tile, and half of the epilogue.
//   warps 8-11  the same for columns 64..127.
// Tensor memory (512 columns): S (0..127) | dP (128..255) | accumulators (256..).  The packed 16-bit
// P / dS of a warpgroup's 64 columns are written over the first 32 columns of that warpgroup's own
// 64 S / dP columns, so no warpgroup overwrites columns the other has yet to read; each K16 step of
// the MMAs that read them addresses its 8 columns directly.
// Every barrier wait gives up after AttnBwdParams::timeout_ns, records bit 0 in this file's device
// status word and stops the CTA after letting its copies and MMAs land.
#include <cuda_runtime.h>
#include <math.h>

#include <type_traits>

#include "attnfuse_internal.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace attnfuse {

__device__ unsigned int g_bwd_status = 0;

namespace {

constexpr int BM = 128;                     // rows per tile (= TMEM lanes)
constexpr int kThreads = 384;
constexpr uint32_t kBoxBytes = 128 * 128;   // 128 rows x 64 16-bit columns, 128-byte swizzled
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t COL_S = 0, COL_DP = 128, COL_ACC = 256;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int NBOX = D / 64;
  static constexpr uint32_t TILE = NBOX * kBoxBytes;
  // Resident pair (dK/dV: K', V; dQ: Q', dO) then a 2-stage ring of pairs (dK/dV: Q', dO; dQ: K', V).
  static constexpr uint32_t OFF_RES = 0;
  static constexpr uint32_t OFF_RING = 2 * TILE;
  static constexpr uint32_t OFF_VEC = OFF_RING + 4 * TILE;  // dK/dV: per stage L[128], D[128] (fp32)
  static constexpr uint32_t OFF_CTL = OFF_VEC + 2 * 2 * BM * 4;
  static constexpr uint32_t SMEM = OFF_CTL + 256 + 1024;
};

struct __align__(8) BwdCtrl {
  uint64_t res_full, res_empty;          // resident pair landed / free again
  uint64_t ring_full[4], ring_empty[2];  // ring stage st, rows 64 h .. 64 h + 63 landed (st * 2 + h) /
                                         // stage free again
  uint64_t s_full[2];                    // S and dP of half h of this step are in tensor memory
  uint64_t p_ready[2];                   // warpgroup h wrote its P / dS (128 arrivals)
  uint64_t acc_full;                     // the unit's accumulators are complete
  uint64_t acc_empty;                    // the epilogue has read them (256 arrivals)
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int skip;
  int unit_slot[8];                      // dQ: unit of the producer's k-th resident load at [k % 8]
};
static_assert(sizeof(BwdCtrl) <= 256, "control block");

__device__ __forceinline__ uint32_t bar_addr(const uint64_t& b) { return ptx::smem_u32(&b); }

__device__ __forceinline__ void signal_abort(BwdCtrl& ctl) {
  *reinterpret_cast<volatile int*>(&ctl.abort_flag) = 1;
  atomicOr(&g_bwd_status, 1u);
}

// Bounded wait on an mbarrier phase; false if this CTA aborted or the wait ran out (then the
// status word and the abort flag are set).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, BwdCtrl& ctl, unsigned long long timeout_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*reinterpret_cast<volatile int*>(&ctl.abort_flag)) return false;
      if (ptx::globaltimer_ns() - t0 > timeout_ns) {
        signal_abort(ctl);
        return false;
      }
    }
  }
}

// Whole-warp form: every lane polls, a vote makes the outcome warp-uniform.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, BwdCtrl& ctl, unsigned long long tmo) {
  return __all_sync(0xFFFFFFFFu, wait_bar(bar, parity, ctl, tmo));
}

// Bounded wait that ignores the abort flag: used only to let in-flight copies and MMAs land.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, unsigned long long timeout_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity))
    if (ptx::globaltimer_ns() - t0 > timeout_ns) return;
}

__device__ __forceinline__ int unit_of_round(int round, int c, int G) {
  return round * G + ((round & 1) ? (G - 1 - c) : c);
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return Pack<BF16>::pack(lo, hi);
}

// D[b, h, i] = dO_i . O_i in fp32.  A thread takes 8 elements (one 16-byte load of each tensor), d/8
// consecutive threads a row, so a warp reads whole 256-byte rows with 16-byte accesses; the group
// reduces with shuffles.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __grid_constant__ AttnBwdParams p) {
  constexpr int TPR = D / 8;  // threads per row: 16 (d = 128) or 8 (d = 64)
  ptx::grid_dep_launch_dependents();
  ptx::grid_dep_wait();  // launched as a dependent of the pre-rotation pass
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (tid == 0) *p.unit_ctr = 0;  // read by the dQ kernel, which starts after this grid completes
  const long long row = tid / TPR;
  const int part = (int)(tid % TPR);
  const long long rows = (long long)p.B * p.N * p.Hq;
  float acc = 0.f;
  if (row < rows) {
    const uint4 ov = *reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(p.out) + (row * D + part * 8) * 2);
    const uint4 gv = *reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(p.dout) + (row * D + part * 8) * 2);
    const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float a0, a1, b0, b1;
      Pack<BF16>::unpack(ow[k], a0, a1);
      Pack<BF16>::unpack(gw[k], b0, b1);
      acc = fmaf(a0, b0, fmaf(a1, b1, acc));
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
  if (row < rows && part == 0) {
    // row = (b * N + i) * Hq + h  ->  D[(b * Hq + h) * N + i]
    const int h = (int)(row % p.Hq);
    const long long bi = row / p.Hq;
    const int i = (int)(bi % p.N);
    const int b = (int)(bi / p.N);
    p.Dvec[((long long)b * p.Hq + h) * p.N + i] = acc;
  }
}

// Causal structure with Nk >= N keys (the N queries are the last N of the Nk tokens: query row i
// sees key j iff j <= q_off + i, q_off = Nk - N).  With q_off = 0 these are key tile kt's first
// query tile kt and query tile t's key tiles 0 .. t.
// First query tile with a row that sees some key of key tile kt.
__device__ __forceinline__ int first_qtile(int kt, const AttnBwdParams& p) {
  const int v = kt * BM - p.q_off;
  return v <= 0 ? 0 : v / BM;
}
// Number of key tiles some row of query tile t sees.
__device__ __forceinline__ int qtile_keytiles(int t, const AttnBwdParams& p) {
  return (p.q_off + min(t * BM + BM - 1, p.N - 1)) / BM + 1;
}

// R(pos)^T applied to the pair (x, y) = (row[e], row[e + d/2]) with frequency F_e.
__device__ __forceinline__ void unrotate_pair(float& x, float& y, uint32_t pos, uint32_t flo, uint32_t fhi) {
  float c, s;
  rope_cs(pos, flo, fhi, c, s);
  const float xr = __fmaf_rn(x, c, __fmul_rn(y, s));
  const float yr = __fmaf_rn(y, c, -__fmul_rn(x, s));
  x = xr;
  y = yr;
}

// S-like product into tensor memory: D[dst] = A B^T with A a 128-row and B a 64-row slice of tiles
// of d columns in shared memory, both K-major (the layout TMA writes; a 64-row slice starts 8 KB
// into each 128-row box).  Consecutive K-steps add a constant to the start address field (offsets
// stay inside the 14-bit field).
template <int D>
__device__ __forceinline__ void issue_kmajor(uint32_t dst, uint32_t a, uint32_t b, uint32_t idesc) {
  const uint64_t da = ptx::sdesc_sw128(a, 16, 1024), db = ptx::sdesc_sw128(b, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t step = (uint64_t)((kk / 4) * (kBoxBytes >> 4) + (kk % 4) * 2);
    ptx::mma_ss_w(dst, da + step, db + step, idesc, kk > 0 ? 1u : 0u);
  }
}

// Accumulation D[dst] (+)= A B with A the packed 16-bit 128 x 128 matrix in tensor memory (K16 step
// kk in the 8 columns at a + 64 (kk / 4) + 8 (kk % 4): each warpgroup's half sits over its own S /
// dP columns) and B a 128-row tile in shared memory read MN-major (N = d columns, K = its rows).
// Only the K-steps of half `half` (K rows [64 half, 64 half + 64)) are issued.
template <int D>
__device__ __forceinline__ void issue_acc(uint32_t dst, uint32_t a, uint32_t b, uint32_t idesc, int half,
                                          bool first) {
  const uint64_t db = ptx::sdesc_sw128(b, kBoxBytes, 1024);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int kk = 4 * half + k;
    ptx::mma_ts_w(dst, a + 64 * (kk / 4) + 8 * (kk % 4), db + (uint64_t)(kk * (2048 >> 4)), idesc,
                  (!first || k > 0) ? 1u : 0u);
  }
}

constexpr uint32_t kHalfRows = 64 * 128;  // byte offset of row 64 inside a 128-row box

// Rows 64 h .. 64 h + 63 of a 128-row tile through a tensor map whose box is 64 rows: they land at
// their place in the tile's swizzled boxes (the 128-byte swizzle repeats every 8 rows).
template <int D>
__device__ __forceinline__ void tma_half(uint32_t tile, const CUtensorMap* map64, uint32_t bar, int head, int row0,
                                         int h, int b) {
#pragma unroll
  for (int bx = 0; bx < D / 64; ++bx)
    ptx::tma_load_4d(tile + bx * kBoxBytes + h * kHalfRows, map64, bar, bx * 64, head, row0 + 64 * h, b);
}

// Common prologue of both kernels: barriers, tensor memory, skip flag.  The dK/dV kernel waits for
// the D kernel and only then lets the dQ kernel launch, so D, q' and k' are complete when the dQ
// kernel starts; the dQ kernel reads nothing the dK/dV kernel writes and runs beside it (its CTAs
// take the SMs the dK/dV CTAs leave), waiting for that grid only before it exits.
template <int D, bool DQ>
__device__ __forceinline__ void bwd_setup(BwdCtrl& ctl, int warp) {
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_addr(ctl.res_full), 1);
    ptx::mbar_init(bar_addr(ctl.res_empty), 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(bar_addr(ctl.ring_full[2 * s]), 1);
      ptx::mbar_init(bar_addr(ctl.ring_full[2 * s + 1]), 1);
      ptx::mbar_init(bar_addr(ctl.ring_empty[s]), 1);
    }
    for (int h = 0; h < 2; ++h) {
      ptx::mbar_init(bar_addr(ctl.s_full[h]), 1);
      ptx::mbar_init(bar_addr(ctl.p_ready[h]), 128);
    }
    ptx::mbar_init(bar_addr(ctl.acc_full), 1);
    ptx::mbar_init(bar_addr(ctl.acc_empty), 256);
    ptx::mbar_init(bar_addr(ctl.mma_done), 1);
    ctl.abort_flag = 0;
    ctl.skip = (*reinterpret_cast<volatile unsigned int*>(&g_bwd_status)) != 0u;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&ctl.tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // Launched as a programmatic dependent of the previous kernel in the chain: the set-up above
  // overlaps its end; nothing it wrote is read before this wait.
  if constexpr (DQ) {
    ptx::grid_dep_launch_dependents();
  } else {
    ptx::grid_dep_wait();
    ptx::grid_dep_launch_dependents();
  }
}

__device__ __forceinline__ void bwd_teardown(BwdCtrl& ctl, int warp, uint32_t tmem) {
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// Let every copy already issued land before shared memory is released.
__device__ __forceinline__ void drain_copies(BwdCtrl& ctl, int res_loads, int ring_loads) {
  const unsigned long long drain = 100000000ull;
  if (res_loads > 0) drain_bar(bar_addr(ctl.res_full), (res_loads - 1) & 1, drain);
  for (int s = 0; s < 2; ++s)
    if (ring_loads > s)
      for (int h = 0; h < 2; ++h) drain_bar(bar_addr(ctl.ring_full[2 * s + h]), ((ring_loads - 1 - s) / 2) & 1, drain);
}

template <int D>
__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar, int head, int row,
                                         int b) {
#pragma unroll
  for (int bx = 0; bx < D / 64; ++bx) ptx::tma_load_4d(dst + bx * kBoxBytes, map, bar, bx * 64, head, row, b);
}

// ================================ dK, dV ==================================================
// Unit u: key tile kt = u / (B Hkv) (ascending, so the units with the most query tiles come first)
// of KV head hk, batch b; steps: query head h of the group (outer), query tile t = kt .. last.
template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const __grid_constant__ AttnBwdParams p) {
  using C = BwdCfg<D>;
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  constexpr uint32_t AB = BF16 ? 1u : 0u;
  constexpr uint32_t IDESC_S = ptx::idesc_f16(AB, BM, 64, 0, 0);  // 128 x 64 halves
  constexpr uint32_t IDESC_ACC = ptx::idesc_f16(AB, BM, D, 0, 1);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);
  BwdCtrl& ctl = *reinterpret_cast<BwdCtrl*>(sgen + C::OFF_CTL);
  const uint32_t sK = sbase + C::OFF_RES, sV = sK + C::TILE, sRing = sbase + C::OFF_RING;
  float* sVec = reinterpret_cast<float*>(sgen + C::OFF_VEC);
  const int warp = __shfl_sync(0xFFFFFFFFu, (int)(threadIdx.x / 32), 0);
  const int lane = threadIdx.x % 32;

  bwd_setup<D, false>(ctl, warp);
  const uint32_t tmem = ctl.tmem_base;
  const bool skip = __shfl_sync(0xFFFFFFFFu, ctl.skip, 0) != 0;
  const unsigned long long tmo = p.timeout_ns;
  const int g = p.Hq / p.Hkv, nt = p.n_tiles, bh_count = p.B * p.Hkv;
  const int total = bh_count * p.n_ktiles;

  if (!skip && warp == 0) {
    // ------------------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmQ);
      ptx::tma_prefetch_desc(&tmK);
      ptx::tma_prefetch_desc(&tmV);
      ptx::tma_prefetch_desc(&tmO);
    }
    int gs = 0, uc = 0;
    bool ok = true;
    for (int rnd = 0; rnd * (int)gridDim.x < total && ok; ++rnd) {
      const int u = unit_of_round(rnd, blockIdx.x, gridDim.x);
      if (u >= total) break;
      const int kt = u / bh_count, bh = u - kt * bh_count, b = bh / p.Hkv, hk = bh - b * p.Hkv;
      if (!(ok = wait_warp(bar_addr(ctl.res_empty), (uc & 1) ^ 1, ctl, tmo))) break;
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(bar_addr(ctl.res_full), 2 * C::TILE);
        tma_tile<D>(sK, &tmK, bar_addr(ctl.res_full), hk, kt * BM, b);
        tma_tile<D>(sV, &tmV, bar_addr(ctl.res_full), hk, kt * BM, b);
      }
      ++uc;
      const int t0 = first_qtile(kt, p), nq = nt - t0;
      for (int s = 0; s < g * nq; ++s) {
        const int h = hk * g + s / nq, t = t0 + s % nq, st = gs & 1;
        // L = lse * log2(e) and D of the tile's 128 query rows (rows past N: L = +inf, so P = 0),
        // read before the stage is free so that their latency overlaps the wait.
        const size_t rbase = ((size_t)b * p.Hq + h) * p.N;
        float lv[4], dv4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int row = t * BM + lane * 4 + k;
          lv[k] = row < p.N ? -(p.lse[rbase + row] * kLog2e) : -INFINITY;  // -L
          dv4[k] = row < p.N ? p.Dvec[rbase + row] : 0.f;
        }
        if (!(ok = wait_warp(bar_addr(ctl.ring_empty[st]), ((gs >> 1) & 1) ^ 1, ctl, tmo))) break;
        float* vL = sVec + st * 2 * BM;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          vL[lane * 4 + k] = lv[k];
          vL[BM + lane * 4 + k] = dv4[k];
        }
        __syncwarp();
        if (lane == 0) {
          // each half of the query rows on its own barrier: the half-steps start as their rows land
          const uint32_t sQ = sRing + st * 2 * C::TILE;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const uint32_t bar = bar_addr(ctl.ring_full[2 * st + hh]);
            ptx::mbar_arrive_expect_tx(bar, C::TILE);
            tma_half<D>(sQ, &tmQ, bar, h, t * BM, hh, b);
            tma_half<D>(sQ + C::TILE, &tmO, bar, h, t * BM, hh, b);
          }
        }
        ++gs;
      }
    }
    if (!ok && lane == 0) drain_copies(ctl, uc, gs);
  } else if (!skip && warp == 1) {
    // ------------------------------------------ MMA issuer --------------------------------
    // Two halves per step (queries 0..63 -> warpgroup 0, 64..127 -> warpgroup 1), software
    // pipelined: S^T, dP^T of one half run on the tensor cores while the other half's warpgroup
    // computes P^T, dS^T.  Order per step g: [dV, dK of half 0 of g] [S^T, dP^T of half 0 of g+1]
    // [dV, dK of half 1 of g] [S^T, dP^T of half 1 of g+1].
    int gs = 0, uc = 0;
    bool ok = true;
    auto issue_s = [&](int g_step, int half) {
      const uint32_t sQ = sRing + (g_step & 1) * 2 * C::TILE + half * kHalfRows, sO = sQ + C::TILE;
      issue_kmajor<D>(tmem + COL_S + 64 * half, sK, sQ, IDESC_S);    // S^T  = K' Q'^T  (64 queries)
      issue_kmajor<D>(tmem + COL_DP + 64 * half, sV, sO, IDESC_S);   // dP^T = V dO^T
      ptx::mma_commit_w(bar_addr(ctl.s_full[half]));
    };
    for (int rnd = 0; rnd * (int)gridDim.x < total && ok; ++rnd) {
      const int u = unit_of_round(rnd, blockIdx.x, gridDim.x);
      if (u >= total) break;
      const int kt = u / bh_count, nsteps = g * (nt - first_qtile(kt, p));
      if (!(ok = wait_warp(bar_addr(ctl.res_full), uc & 1, ctl, tmo))) break;
      for (int half = 0; half < 2 && ok; ++half) {
        if (!(ok = wait_warp(bar_addr(ctl.ring_full[2 * (gs & 1) + half]), (gs >> 1) & 1, ctl, tmo))) break;
        ptx::tc_fence_after();
        issue_s(gs, half);
      }
      if (!ok) break;
      for (int s = 0; s < nsteps; ++s) {
        const int st = gs & 1;
        const uint32_t sQ = sRing + st * 2 * C::TILE, sO = sQ + C::TILE;
        const bool more = s + 1 < nsteps;
        for (int half = 0; half < 2; ++half) {
          if (!(ok = wait_warp(bar_addr(ctl.p_ready[half]), gs & 1, ctl, tmo))) break;
          if (s == 0 && half == 0 && uc > 0 && !(ok = wait_warp(bar_addr(ctl.acc_empty), (uc - 1) & 1, ctl, tmo)))
            break;
          ptx::tc_fence_after();
          const bool first = s == 0 && half == 0;
          issue_acc<D>(tmem + COL_ACC, tmem + COL_S, sO, IDESC_ACC, half, first);       // dV  += P^T dO
          issue_acc<D>(tmem + COL_ACC + D, tmem + COL_DP, sQ, IDESC_ACC, half, first);  // dK' += dS^T Q'
          if (half == 1) ptx::mma_commit_w(bar_addr(ctl.ring_empty[st]));
          if (more) {
            if (!(ok = wait_warp(bar_addr(ctl.ring_full[2 * ((gs + 1) & 1) + half]), ((gs + 1) >> 1) & 1, ctl, tmo)))
              break;
            ptx::tc_fence_after();
            issue_s(gs + 1, half);
          }
        }
        if (!ok) break;
        ++gs;
      }
      if (!ok) break;
      ptx::mma_commit_w(bar_addr(ctl.acc_full));
      ptx::mma_commit_w(bar_addr(ctl.res_empty));
      ++uc;
    }
    ptx::mma_commit_w(bar_addr(ctl.mma_done));
    drain_bar(bar_addr(ctl.mma_done), 0, 100000000ull);
  } else if (!skip && warp >= 4) {
    // ------------------------------------------ elementwise + epilogue --------------------
    const int wg = (warp - 4) / 4;             // query columns [64 wg, 64 wg + 64)
    const int r = (warp & 3) * 32 + lane;      // key row in the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + COL_S, tP = tmem + lane_off + COL_DP, tA = tmem + lane_off + COL_ACC;
    const uint64_t sl2x2 = ptx::f2_pack(p.scale_log2, p.scale_log2);
    int gs = 0, uc = 0;
    bool ok = true;
    for (int rnd = 0; rnd * (int)gridDim.x < total && ok; ++rnd) {
      const int u = unit_of_round(rnd, blockIdx.x, gridDim.x);
      if (u >= total) break;
      const int kt = u / bh_count, bh = u - kt * bh_count, b = bh / p.Hkv, hk = bh - b * p.Hkv;
      const int t0 = first_qtile(kt, p), nq = nt - t0;
      for (int s = 0; s < g * nq; ++s) {
        const int t = t0 + s % nq, st = gs & 1;
        if (!(ok = wait_warp(bar_addr(ctl.s_full[wg]), gs & 1, ctl, tmo))) break;
        if (!(ok = wait_warp(bar_addr(ctl.ring_full[2 * st + wg]), (gs >> 1) & 1, ctl, tmo))) break;
        ptx::tc_fence_after();
        const float* vL = sVec + st * 2 * BM;
        // query c of the tile sees key r iff c >= r - delta; only tiles with delta < 127 mask anything
        const int delta = p.q_off + (t - kt) * BM;
        const bool diag = delta < BM - 1;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int q0 = 64 * wg + 32 * c;
          uint32_t sv[32], dv[32];
          ptx::tmem_ld32(tS + q0, sv);
          ptx::tmem_ld32(tP + q0, dv);
          ptx::tmem_wait_ld();
          uint32_t pp[16], dsp[16];
          // Column pairs in fp32x2 arithmetic (the same IEEE operations): P = 2^(S sl2 - L),
          // dS = P (dP - D); the vectors hold -L and D.
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int q = q0 + 2 * e;
            float x0, x1;
            ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), sl2x2,
                                       *reinterpret_cast<const uint64_t*>(vL + q)),
                           x0, x1);
            float p0 = ptx::ex2_approx(x0), p1 = ptx::ex2_approx(x1);
            if (diag) {
              if (q < r - delta) p0 = 0.f;
              if (q + 1 < r - delta) p1 = 0.f;
            }
            const uint64_t dd = ptx::f2_sub(ptx::f2_pack(__uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1])),
                                            *reinterpret_cast<const uint64_t*>(vL + BM + q));
            float d0, d1;
            ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(p0, p1), dd), d0, d1);
            pp[e] = pack2<BF16>(p0, p1);
            dsp[e] = pack2<BF16>(d0, d1);
          }
          ptx::tmem_st16(tS + 64 * wg + 16 * c, pp);
          ptx::tmem_st16(tP + 64 * wg + 16 * c, dsp);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_addr(ctl.p_ready[wg]));
        ++gs;
      }
      if (!ok) break;
      // Epilogue: dV columns [wg d/2, wg d/2 + d/2); dK' pairs e in [wg d/4, wg d/4 + d/4) with e + d/2.
      if (!(ok = wait_warp(bar_addr(ctl.acc_full), uc & 1, ctl, tmo))) break;
      ptx::tc_fence_after();
      constexpr int HV = D / 2, QK = D / 4;
      uint32_t vv[HV], kx[QK], ky[QK];
#pragma unroll
      for (int c = 0; c < HV / 32; ++c) {
        uint32_t tmp[32];
        ptx::tmem_ld32(tA + wg * HV + 32 * c, tmp);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) vv[32 * c + e] = tmp[e];
      }
      if constexpr (QK == 32) {
        ptx::tmem_ld32(tA + D + wg * QK, kx);
        ptx::tmem_ld32(tA + D + HV + wg * QK, ky);
      } else {
        ptx::tmem_ld16(tA + D + wg * QK, kx);
        ptx::tmem_ld16(tA + D + HV + wg * QK, ky);
      }
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar_addr(ctl.acc_empty));
      ++uc;
      const int j = kt * BM + r;
      if (j < p.Nk) {
        T* dvrow = reinterpret_cast<T*>(p.dv) + (((size_t)b * p.Nk + j) * p.Hkv + hk) * D;
        T* dkrow = reinterpret_cast<T*>(p.dk) + (((size_t)b * p.Nk + j) * p.Hkv + hk) * D;
#pragma unroll
        for (int v = 0; v < HV / 8; ++v) {
          uint4 w;
          w.x = pack2<BF16>(__uint_as_float(vv[8 * v]), __uint_as_float(vv[8 * v + 1]));
          w.y = pack2<BF16>(__uint_as_float(vv[8 * v + 2]), __uint_as_float(vv[8 * v + 3]));
          w.z = pack2<BF16>(__uint_as_float(vv[8 * v + 4]), __uint_as_float(vv[8 * v + 5]));
          w.w = pack2<BF16>(__uint_as_float(vv[8 * v + 6]), __uint_as_float(vv[8 * v + 7]));
          *reinterpret_cast<uint4*>(dvrow + wg * HV + 8 * v) = w;
        }
        float x[QK], y[QK];
#pragma unroll
        for (int e = 0; e < QK; ++e) {
          x[e] = __uint_as_float(kx[e]) * p.inv_sqrt_d;
          y[e] = __uint_as_float(ky[e]) * p.inv_sqrt_d;
          const int k = wg * QK + e;
          if (p.unrotate) unrotate_pair(x[e], y[e], (uint32_t)j, p.freqs.lo[k], p.freqs.hi[k]);
        }
#pragma unroll
        for (int v = 0; v < QK / 8; ++v) {
          uint4 wx, wy;
          wx.x = pack2<BF16>(x[8 * v], x[8 * v + 1]);
          wx.y = pack2<BF16>(x[8 * v + 2], x[8 * v + 3]);
          wx.z = pack2<BF16>(x[8 * v + 4], x[8 * v + 5]);
          wx.w = pack2<BF16>(x[8 * v + 6], x[8 * v + 7]);
          wy.x = pack2<BF16>(y[8 * v], y[8 * v + 1]);
          wy.y = pack2<BF16>(y[8 * v + 2], y[8 * v + 3]);
          wy.z = pack2<BF16>(y[8 * v + 4], y[8 * v + 5]);
          wy.w = pack2<BF16>(y[8 * v + 6], y[8 * v + 7]);
          *reinterpret_cast<uint4*>(dkrow + wg * QK + 8 * v) = wx;
          *reinterpret_cast<uint4*>(dkrow + HV + wg * QK + 8 * v) = wy;
        }
      }
    }
  }
  bwd_teardown(ctl, warp, tmem);
}

// ================================ dQ ======================================================
// Unit u: query tile t = nt - 1 - u / (B Hq) (descending: the longest units first) of head h, batch
// b; steps: the key tiles j of KV head h / g that some row of the tile sees (0 .. t when N == Nk).
// Units are handed out in that order by a global counter: the producer takes the next one when it
// has room for a resident pair and publishes it in the control block before the pair's copies
// (the resident barrier's completion makes it visible to the other roles); a CTA that starts late,
// on an SM a dK/dV CTA has just left, simply takes fewer units.  A value >= the unit count, posted
// with a copy-less arrival on the resident barrier, ends every role.
template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const __grid_constant__ AttnBwdParams p) {
  using C = BwdCfg<D>;
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  constexpr uint32_t AB = BF16 ? 1u : 0u;
  constexpr uint32_t IDESC_S = ptx::idesc_f16(AB, BM, 64, 0, 0);  // 128 x 64 halves
  constexpr uint32_t IDESC_ACC = ptx::idesc_f16(AB, BM, D, 0, 1);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);
  BwdCtrl& ctl = *reinterpret_cast<BwdCtrl*>(sgen + C::OFF_CTL);
  const uint32_t sQ = sbase + C::OFF_RES, sO = sQ + C::TILE, sRing = sbase + C::OFF_RING;
  float* sVec = reinterpret_cast<float*>(sgen + C::OFF_VEC);  // this unit's L[128], D[128] (fp32)
  const int warp = __shfl_sync(0xFFFFFFFFu, (int)(threadIdx.x / 32), 0);
  const int lane = threadIdx.x % 32;

  bwd_setup<D, true>(ctl, warp);
  const uint32_t tmem = ctl.tmem_base;
  const bool skip = __shfl_sync(0xFFFFFFFFu, ctl.skip, 0) != 0;
  const unsigned long long tmo = p.timeout_ns;
  const int g = p.Hq / p.Hkv, nt = p.n_tiles, bh_count = p.B * p.Hq;
  const int total = bh_count * nt;

  if (!skip && warp == 0) {
    // ------------------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmQ);
      ptx::tma_prefetch_desc(&tmK);
      ptx::tma_prefetch_desc(&tmV);
      ptx::tma_prefetch_desc(&tmO);
    }
    int gs = 0, uc = 0;
    bool ok = true;
    // Each unit is taken from the counter one unit ahead, and its rows' L = lse * log2(e) and D are
    // read before the resident buffers are free: neither round trip sits between the previous
    // unit's last product and this unit's copies.  The vectors go to shared memory with the unit.
    int u_next = 0;
    if (lane == 0) u_next = atomicAdd(p.unit_ctr, 1);
    u_next = __shfl_sync(0xFFFFFFFFu, u_next, 0);
    for (;;) {
      const int u = u_next;
      float lv[4], dv4[4];
      if (u < total) {
        if (lane == 0) u_next = atomicAdd(p.unit_ctr, 1);
        u_next = __shfl_sync(0xFFFFFFFFu, u_next, 0);
        const int t_ = nt - 1 - u / bh_count, bh_ = u % bh_count, b_ = bh_ / p.Hq, h_ = bh_ - b_ * p.Hq;
        const size_t rbase = ((size_t)b_ * p.Hq + h_) * p.N;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int row = t_ * BM + lane * 4 + k;
          lv[k] = row < p.N ? p.lse[rbase + row] * kLog2e : INFINITY;  // rows past N: P = 0
          dv4[k] = row < p.N ? p.Dvec[rbase + row] : 0.f;
        }
      }
      if (!(ok = wait_warp(bar_addr(ctl.res_empty), (uc & 1) ^ 1, ctl, tmo))) break;
      if (u >= total) {
        if (lane == 0) {
          ctl.unit_slot[uc & 7] = total;
          ptx::mbar_arrive(bar_addr(ctl.res_full));
        }
        break;
      }
      const int t = nt - 1 - u / bh_count, bh = u % bh_count, b = bh / p.Hq, h = bh - b * p.Hq;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        sVec[lane * 4 + k] = lv[k];
        sVec[BM + lane * 4 + k] = dv4[k];
      }
      __syncwarp();
      if (lane == 0) {
        ctl.unit_slot[uc & 7] = u;
        ptx::mbar_arrive_expect_tx(bar_addr(ctl.res_full), 2 * C::TILE);
        tma_tile<D>(sQ, &tmQ, bar_addr(ctl.res_full), h, t * BM, b);
        tma_tile<D>(sO, &tmO, bar_addr(ctl.res_full), h, t * BM, b);
      }
      ++uc;
      for (int j = 0, nkj = qtile_keytiles(t, p); j < nkj; ++j) {
        const int st = gs & 1;
        if (!(ok = wait_warp(bar_addr(ctl.ring_empty[st]), ((gs >> 1) & 1) ^ 1, ctl, tmo))) break;
        if (lane == 0) {
          // each half of the key rows on its own barrier
          const uint32_t sK = sRing + st * 2 * C::TILE;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const uint32_t bar = bar_addr(ctl.ring_full[2 * st + hh]);
            ptx::mbar_arrive_expect_tx(bar, C::TILE);
            tma_half<D>(sK, &tmK, bar, h / g, j * BM, hh, b);
            tma_half<D>(sK + C::TILE, &tmV, bar, h / g, j * BM, hh, b);
          }
        }
        ++gs;
      }
    }
    if (!ok && lane == 0) drain_copies(ctl, uc, gs);
  } else if (!skip && warp == 1) {
    // ------------------------------------------ MMA issuer --------------------------------
    // Two halves per key tile (keys 0..63 -> warpgroup 0, 64..127 -> warpgroup 1), pipelined as in
    // the dK/dV kernel: [dQ' += dS K' of half 0 of j] [S, dP of half 0 of j+1] [half 1 of j] ...
    int gs = 0, uc = 0;
    bool ok = true;
    auto issue_s = [&](int g_step, int half) {
      const uint32_t sK = sRing + (g_step & 1) * 2 * C::TILE + half * kHalfRows, sV = sK + C::TILE;
      issue_kmajor<D>(tmem + COL_S + 64 * half, sQ, sK, IDESC_S);   // S  = Q' K'^T  (64 keys)
      issue_kmajor<D>(tmem + COL_DP + 64 * half, sO, sV, IDESC_S);  // dP = dO V^T
      ptx::mma_commit_w(bar_addr(ctl.s_full[half]));
    };
    for (;;) {
      if (!(ok = wait_warp(bar_addr(ctl.res_full), uc & 1, ctl, tmo))) break;
      const int u = *reinterpret_cast<volatile int*>(&ctl.unit_slot[uc & 7]);
      if (u >= total) break;
      const int t = nt - 1 - u / bh_count;
      for (int half = 0; half < 2 && ok; ++half) {
        if (!(ok = wait_warp(bar_addr(ctl.ring_full[2 * (gs & 1) + half]), (gs >> 1) & 1, ctl, tmo))) break;
        ptx::tc_fence_after();
        issue_s(gs, half);
      }
      if (!ok) break;
      const int nkj = qtile_keytiles(t, p);
      for (int j = 0; j < nkj; ++j) {
        const int st = gs & 1;
        const uint32_t sK = sRing + st * 2 * C::TILE;
        const bool more = j + 1 < nkj;
        for (int half = 0; half < 2; ++half) {
          if (!(ok = wait_warp(bar_addr(ctl.p_ready[half]), gs & 1, ctl, tmo))) break;
          if (j == 0 && half == 0 && uc > 0 && !(ok = wait_warp(bar_addr(ctl.acc_empty), (uc - 1) & 1, ctl, tmo)))
            break;
          ptx::tc_fence_after();
          issue_acc<D>(tmem + COL_ACC, tmem + COL_S, sK, IDESC_ACC, half, j == 0 && half == 0);  // dQ' += dS K'
          if (half == 1) ptx::mma_commit_w(bar_addr(ctl.ring_empty[st]));
          if (more) {
            if (!(ok = wait_warp(bar_addr(ctl.ring_full[2 * ((gs + 1) & 1) + half]), ((gs + 1) >> 1) & 1, ctl, tmo)))
              break;
            ptx::tc_fence_after();
            issue_s(gs + 1, half);
          }
        }
        if (!ok) break;
        ++gs;
      }
      if (!ok) break;
      ptx::mma_commit_w(bar_addr(ctl.acc_full));
      ptx::mma_commit_w(bar_addr(ctl.res_empty));
      ++uc;
    }
    ptx::mma_commit_w(bar_addr(ctl.mma_done));
    drain_bar(bar_addr(ctl.mma_done), 0, 100000000ull);
  } else if (!skip && warp >= 4) {
    // ------------------------------------------ elementwise + epilogue --------------------
    const int wg = (warp - 4) / 4;             // key columns [64 wg, 64 wg + 64)
    const int r = (warp & 3) * 32 + lane;      // query row in the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + COL_S, tP = tmem + lane_off + COL_DP, tA = tmem + lane_off + COL_ACC;
    const uint64_t sl2x2 = ptx::f2_pack(p.scale_log2, p.scale_log2);
    int gs = 0, uc = 0;
    bool ok = true;
    for (;;) {
      if (!(ok = wait_warp(bar_addr(ctl.res_full), uc & 1, ctl, tmo))) break;
      const int u = *reinterpret_cast<volatile int*>(&ctl.unit_slot[uc & 7]);
      if (u >= total) break;
      const int t = nt - 1 - u / bh_count, bh = u % bh_count, b = bh / p.Hq, h = bh - b * p.Hq;
      const int i = t * BM + r;
      const float L = sVec[r], Dr = sVec[BM + r];  // staged by the producer with the unit
      const uint64_t nl2 = ptx::f2_pack(-L, -L), dr2 = ptx::f2_pack(Dr, Dr);
      const int nkj = qtile_keytiles(t, p);
      for (int j = 0; j < nkj; ++j) {
        if (!(ok = wait_warp(bar_addr(ctl.s_full[wg]), gs & 1, ctl, tmo))) break;
        ptx::tc_fence_after();
        // key c of the tile is visible to query r iff c <= r + delta; only tiles with delta < 127 mask
        const int delta = p.q_off + (t - j) * BM;
        const bool diag = delta < BM - 1;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int k0 = 64 * wg + 32 * c;
          uint32_t sv[32], dv[32];
          ptx::tmem_ld32(tS + k0, sv);
          ptx::tmem_ld32(tP + k0, dv);
          ptx::tmem_wait_ld();
          uint32_t dsp[16];
          // Column pairs in fp32x2 arithmetic (the same IEEE operations): P = 2^(S sl2 - L), dS = P (dP - D).
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int k = k0 + 2 * e;
            float x0, x1;
            ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), sl2x2, nl2),
                           x0, x1);
            float p0 = ptx::ex2_approx(x0), p1 = ptx::ex2_approx(x1);
            if (diag) {
              if (k > r + delta) p0 = 0.f;
              if (k + 1 > r + delta) p1 = 0.f;
            }
            const uint64_t dd = ptx::f2_sub(ptx::f2_pack(__uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1])), dr2);
            float d0, d1;
            ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(p0, p1), dd), d0, d1);
            dsp[e] = pack2<BF16>(d0, d1);
          }
          ptx::tmem_st16(tS + 64 * wg + 16 * c, dsp);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_addr(ctl.p_ready[wg]));
        ++gs;
      }
      if (!ok) break;
      // Epilogue: dQ' pairs e in [wg d/4, wg d/4 + d/4) with e + d/2.
      if (!(ok = wait_warp(bar_addr(ctl.acc_full), uc & 1, ctl, tmo))) break;
      ptx::tc_fence_after();
      constexpr int HV = D / 2, QK = D / 4;
      uint32_t qx[QK], qy[QK];
      if constexpr (QK == 32) {
        ptx::tmem_ld32(tA + wg * QK, qx);
        ptx::tmem_ld32(tA + HV + wg * QK, qy);
      } else {
        ptx::tmem_ld16(tA + wg * QK, qx);
        ptx::tmem_ld16(tA + HV + wg * QK, qy);
      }
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar_addr(ctl.acc_empty));
      ++uc;
      if (i < p.N) {
        T* dqrow = reinterpret_cast<T*>(p.dq) + (((size_t)b * p.N + i) * p.Hq + h) * D;
        float x[QK], y[QK];
#pragma unroll
        for (int e = 0; e < QK; ++e) {
          x[e] = __uint_as_float(qx[e]) * p.inv_sqrt_d;
          y[e] = __uint_as_float(qy[e]) * p.inv_sqrt_d;
          const int k = wg * QK + e;
          if (p.unrotate) unrotate_pair(x[e], y[e], (uint32_t)(p.q_off + i), p.freqs.lo[k], p.freqs.hi[k]);
        }
#pragma unroll
        for (int v = 0; v < QK / 8; ++v) {
          uint4 wx, wy;
          wx.x = pack2<BF16>(x[8 * v], x[8 * v + 1]);
          wx.y = pack2<BF16>(x[8 * v + 2], x[8 * v + 3]);
          wx.z = pack2<BF16>(x[8 * v + 4], x[8 * v + 5]);
          wx.w = pack2<BF16>(x[8 * v + 6], x[8 * v + 7]);
          wy.x = pack2<BF16>(y[8 * v], y[8 * v + 1]);
          wy.y = pack2<BF16>(y[8 * v + 2], y[8 * v + 3]);
          wy.z = pack2<BF16>(y[8 * v + 4], y[8 * v + 5]);
          wy.w = pack2<BF16>(y[8 * v + 6], y[8 * v + 7]);
          *reinterpret_cast<uint4*>(dqrow + wg * QK + 8 * v) = wx;
          *reinterpret_cast<uint4*>(dqrow + HV + wg * QK + 8 * v) = wy;
        }
      }
    }
  }
  bwd_teardown(ctl, warp, tmem);
  // The grid completes only after the dK/dV grid it ran beside, so whatever follows on the stream
  // (the pass that rotates dq and dk back, the caller's work) sees both gradients.
  ptx::grid_dep_wait();
}

// Launch as a programmatic dependent of the previous kernel on the stream (it waits in-kernel).
template <typename K, typename... Args>
cudaError_t launch_dependent(K kernel, dim3 grid, dim3 block, uint32_t smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// One CTA per SM (shared memory admits one), each walking its share of the units.  TAG separates
// the per-device set-up caches of kernels that share a signature.
template <int TAG, typename K>
cudaError_t launch_persistent(K kernel, uint32_t smem, int units, const CUtensorMap& mq, const CUtensorMap& mk,
                              const CUtensorMap& mv, const CUtensorMap& mo, const AttnBwdParams& p,
                              cudaStream_t stream) {
  static DeviceOnce once;  // attributes set and SM count kept per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = once.get(dev, [&](int* out) -> cudaError_t {
    cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (r != cudaSuccess) return r;
    return cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
  }, &sms);
  if (e != cudaSuccess) return e;
  const int grid = units < sms ? units : sms;
  return launch_dependent(kernel, dim3((unsigned)grid), dim3(kThreads), smem, stream, mq, mk, mv, mo, p);
}

template <int D, bool BF16>
cudaError_t launch_bwd_impl(const AttnBwdMaps& m, const AttnBwdParams& p, cudaStream_t stream) {
  const long long rows = (long long)p.B * p.N * p.Hq;
  const long long blocks = (rows * (D / 8) + 255) / 256;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  cudaError_t e = launch_dependent(bwd_prep_kernel<D, BF16>, dim3((unsigned)blocks), dim3(256), 0, stream, p);
  if (e != cudaSuccess) return e;
  // the dK/dV kernel streams q', dout in 64-row halves; the dQ kernel streams k', v in 64-row halves
  e = launch_persistent<2 * D + BF16 * 1>(bwd_dkdv_kernel<D, BF16>, BwdCfg<D>::SMEM, p.B * p.Hkv * p.n_ktiles, m.q64,
                                          m.k, m.v, m.dout64, p, stream);
  if (e != cudaSuccess) return e;
  return launch_persistent<2 * D + BF16 * 1 + 1000>(bwd_dq_kernel<D, BF16>, BwdCfg<D>::SMEM, p.B * p.Hq * p.n_tiles,
                                                   m.q, m.k64, m.v64, m.dout, p, stream);
}

}  // namespace

cudaError_t launch_attn_bwd(const AttnBwdMaps& maps, const AttnBwdParams& p, int d, bool bf16, cudaStream_t stream) {
  if (p.n_tiles <= 0) return cudaSuccess;
  if (d == 128) return bf16 ? launch_bwd_impl<128, true>(maps, p, stream) : launch_bwd_impl<128, false>(maps, p, stream);
  return bf16 ? launch_bwd_impl<64, true>(maps, p, stream) : launch_bwd_impl<64, false>(maps, p, stream);
}

cudaError_t read_and_clear_bwd_status(unsigned int* value) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_bwd_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  if (*value != 0u) {
    const unsigned int zero = 0u;
    e = cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace attnfuse
