// The C ABI of libattnfuse: argument validation, device checks, TMA descriptors, workspace
// handling and the launch sequence of each mode.  Declared in include/attnfuse.h.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "attnfuse.h"
#include "attnfuse_internal.h"

namespace attnfuse {

namespace {

// F_k = round(theta_k / (2 pi) * 2^64): frequency of pair k in turns per position, as a 64-bit
// fixed-point fraction (theta_k <= 1, so F_k < 2^61.4).  theta_k = base^(-2k/d) in double.
void compute_freqs(int r, double base, RopeFreqs* f) {
  std::memset(f, 0, sizeof(*f));
  const double two_pi = 6.283185307179586476925286766559;
  for (int k = 0; k < r / 2 && k < kMaxHalfDim; ++k) {
    const double theta = std::pow(base, -2.0 * (double)k / (double)r);
    const double scaled = std::ldexp(theta / two_pi, 64);
    const uint64_t F = (uint64_t)std::llround(scaled);  // < 2^62: fits a signed 64-bit round
    f->lo[k] = (uint32_t)(F & 0xFFFFFFFFull);
    f->hi[k] = (uint32_t)(F >> 32);
  }
}

}  // namespace

// The table for (r, base), from a per-thread cache of the last few pairs asked for (a call
// otherwise spends 32-64 pow() evaluations on it).  Per thread, so no lock is taken.
void rope_freqs_host(int r, double base, RopeFreqs* f) {
  struct Entry {
    int r;
    double base;
    RopeFreqs f;
  };
  constexpr int kEntries = 4;
  thread_local Entry cache[kEntries];
  thread_local int used = 0, next = 0;
  for (int i = 0; i < used; ++i)
    if (cache[i].r == r && cache[i].base == base) {
      *f = cache[i].f;
      return;
    }
  compute_freqs(r, base, f);
  cache[next] = Entry{r, base, *f};
  next = (next + 1) % kEntries;
  if (used < kEntries) ++used;
}

}  // namespace attnfuse

namespace {

using namespace attnfuse;

constexpr unsigned long long kTimeoutNs = 1000000000ull;  // 1 s on any single barrier wait
constexpr int kMaxN = 1 << 24;

thread_local char g_err[512] = "";

attnfuse_status_t fail(attnfuse_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return st;
}

attnfuse_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(ATTNFUSE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

attnfuse_status_t check_dtype_d(int d, attnfuse_dtype_t dtype) {
  if (dtype != ATTNFUSE_BF16 && dtype != ATTNFUSE_FP16) return fail(ATTNFUSE_ERR_INVALID_ARG, "dtype %d is not bf16 (0) or fp16 (1)", (int)dtype);
  if (d != 64 && d != 128) return fail(ATTNFUSE_ERR_UNSUPPORTED, "head dim d=%d is not supported (64 or 128)", d);
  return ATTNFUSE_OK;
}

attnfuse_status_t check_base(double base) {
  if (!(base > 1.0) || !std::isfinite(base)) return fail(ATTNFUSE_ERR_INVALID_ARG, "rope_base must be finite and > 1");
  return ATTNFUSE_OK;
}

// The kernels are built for sm_103a only.  A device's compute capability is queried once and the
// answer kept (0 = not yet known, else major * 10 + minor); concurrent first calls may both query,
// which is harmless.
constexpr int kMaxDevices = 64;
std::atomic<int> g_device_cc[kMaxDevices];

attnfuse_status_t check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTNFUSE_ERR_UNSUPPORTED, "device index %d is beyond %d", dev, kMaxDevices);
  int cc = g_device_cc[dev].load(std::memory_order_acquire);
  if (cc == 0) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    cc = major * 10 + minor;
    g_device_cc[dev].store(cc, std::memory_order_release);
  }
  if (cc != 103)
    return fail(ATTNFUSE_ERR_UNSUPPORTED, "device %d has compute capability %d.%d; libattnfuse runs on 10.3 (sm_103a)",
                dev, cc / 10, cc % 10);
  return ATTNFUSE_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [B, N, H, d] tensor, boxes of 64 columns x 128 rows of one head, 128-byte swizzle.  A descriptor
// depends only on the address, the sizes and the dtype, so the last few encoded are kept per thread
// (a repeated call then encodes nothing; no lock is taken).
attnfuse_status_t encode_bnhd_uncached(CUtensorMap* map, const void* ptr, int B, int N, int H, int d,
                                       attnfuse_dtype_t dtype, int box_rows, const char* name);

// box_rows: tokens per box (128 for the attention tiles, 64 for the half tiles the backward streams, 16
// for the decode kernel's key chunks).
attnfuse_status_t encode_bnhd(CUtensorMap* map, const void* ptr, int B, int N, int H, int d, attnfuse_dtype_t dtype,
                              const char* name, int box_rows = 128) {
  struct Entry {
    const void* ptr;
    int B, N, H, d, box_rows;
    attnfuse_dtype_t dtype;
    CUtensorMap map;
  };
  constexpr int kEntries = 16;
  thread_local Entry cache[kEntries];
  thread_local int used = 0, next = 0;
  for (int i = 0; i < used; ++i) {
    const Entry& c = cache[i];
    if (c.ptr == ptr && c.B == B && c.N == N && c.H == H && c.d == d && c.box_rows == box_rows && c.dtype == dtype) {
      *map = c.map;
      return ATTNFUSE_OK;
    }
  }
  const attnfuse_status_t st = encode_bnhd_uncached(map, ptr, B, N, H, d, dtype, box_rows, name);
  if (st != ATTNFUSE_OK) return st;
  cache[next] = Entry{ptr, B, N, H, d, box_rows, dtype, *map};
  next = (next + 1) % kEntries;
  if (used < kEntries) ++used;
  return ATTNFUSE_OK;
}

attnfuse_status_t encode_bnhd_uncached(CUtensorMap* map, const void* ptr, int B, int N, int H, int d,
                                       attnfuse_dtype_t dtype, int box_rows, const char* name) {
  auto fn = encode_fn();
  if (!fn) return fail(ATTNFUSE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2, (cuuint64_t)N * H * d * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, dtype == ATTNFUSE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                  const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTNFUSE_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name, (int)r);
  return ATTNFUSE_OK;
}

size_t tensor_bytes(int B, int N, int H, int d) { return (size_t)B * (size_t)N * (size_t)H * (size_t)d * 2u; }

// Few queries per KV head (decode, speculative decode): the split-KV decode kernels serve FUSED and
// AUTO calls with at most 16 query rows (rows = (Hq / Hkv) N) per KV head, one MMA tile of rows.
// Measured on GB300 (d = 128, bf16, Llama heads 32/8): faster than the tile kernels at every
// batch tried, from B = 1 (26 vs 62 us over 4096 keys, 68 vs 386 us over 32768) to B = 64 (405 vs
// 488 us), and with 16 rows up to B Hkv = 128 (142 vs 150 us).
bool decode_eligible(int B, int Hq, int Hkv, int N, attnfuse_mode_t mode) {
  if (mode != ATTNFUSE_FUSED && mode != ATTNFUSE_AUTO) return false;
  const long long rows = (long long)(Hq / Hkv) * N;
  return rows <= kDecodeMaxRows && B <= 65535 && Hkv <= 65535;  // grid limits
}

// Splits of the keys, in 16-key chunks: the number of slices that minimises (waves of CTAs) x
// (chunks per warp of a slice + a CTA's fixed work, about three chunks' time) with
// decode_ctas_per_sm(d) CTAs resident per SM on 152 SMs and decode_warps(B, Hkv, d, rows) warps per
// CTA, fewest slices among equals (each slice adds a partial to merge).  A slice count rounded up
// past a whole wave would double the time.
void decode_plan(int B, int Hkv, int Nk, int d, int rows, int* keys_per_split, int* n_splits) {
  const int warps = decode_warps(B, Hkv, d, rows);
  const long long kSlots = 152LL * decode_ctas_per_sm(d);
  constexpr long long kFixedChunks = 3;
  const int chunks = (Nk + kDecodeChunk - 1) / kDecodeChunk;
  const long long heads = (long long)B * Hkv;
  long long best_cost = -1;
  int best_per = chunks;
  const int max_splits = chunks < 1024 ? chunks : 1024;
  for (int s = 1; s <= max_splits; ++s) {
    const int per = (chunks + s - 1) / s;
    const long long n = (chunks + per - 1) / per;  // slices actually needed
    const long long waves = (heads * n + kSlots - 1) / kSlots;
    const long long cost = waves * ((per + warps - 1) / warps + kFixedChunks);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_per = per;
    }
  }
  *keys_per_split = kDecodeChunk * best_per;
  *n_splits = (Nk + *keys_per_split - 1) / *keys_per_split;
}

size_t decode_workspace_bytes(int B, int Hkv, int Nk, int d, int rows) {
  int kps = 0, ns = 0;
  decode_plan(B, Hkv, Nk, d, rows, &kps, &ns);
  const size_t slots = (size_t)B * Hkv * ns * kDecodeMaxRows;
  return round_up(slots * d * sizeof(float), 256) + round_up(slots * 2 * sizeof(float), 256);
}

// The options of an _ex call with their defaults filled in.
struct Opts {
  int rdim;        // rotary dimension (0 -> d)
  int interleaved;
  int Nk;          // key/value tokens (0 -> N)
  const int32_t* qpos;
  const int32_t* kpos;
};

// Resolves and checks the options: r in [16, d], r % 16 == 0; interleaved 0/1; N <= Nk < 2^24;
// position arrays 4-byte aligned.
attnfuse_status_t resolve_opts(const attnfuse_rope_opts_t* o, int d, int N, Opts* x) {
  x->rdim = (o && o->rotary_dim) ? o->rotary_dim : d;
  x->interleaved = o ? o->interleaved : 0;
  x->Nk = (o && o->kv_len) ? o->kv_len : N;
  x->qpos = o ? o->q_positions : nullptr;
  x->kpos = o ? o->k_positions : nullptr;
  if (x->rdim < 16 || x->rdim > d || (x->rdim % 16) != 0)
    return fail(ATTNFUSE_ERR_INVALID_ARG, "rotary_dim=%d must be 0 or a multiple of 16 in [16, d=%d]", x->rdim, d);
  if (x->interleaved != 0 && x->interleaved != 1)
    return fail(ATTNFUSE_ERR_INVALID_ARG, "interleaved=%d must be 0 or 1", x->interleaved);
  if (x->Nk < N || x->Nk >= kMaxN)
    return fail(ATTNFUSE_ERR_INVALID_ARG, "kv_len=%d must be 0 or in [N=%d, %d]", o ? o->kv_len : 0, N, kMaxN - 1);
  if ((x->qpos && !aligned(x->qpos, 4)) || (x->kpos && !aligned(x->kpos, 4)))
    return fail(ATTNFUSE_ERR_INVALID_ARG, "q_positions and k_positions must be 4-byte aligned");
  return ATTNFUSE_OK;
}

attnfuse_status_t validate_fwd(const void* q, const void* k, const void* v, const void* out, const float* lse, int B,
                               int Hq, int Hkv, int N, int d, double base, attnfuse_mode_t mode,
                               attnfuse_dtype_t dtype) {
  if (!q || !k || !v || !out) return fail(ATTNFUSE_ERR_INVALID_ARG, "q, k, v and out must be non-null");
  if (B < 1 || Hq < 1 || Hkv < 1 || N < 1) return fail(ATTNFUSE_ERR_INVALID_ARG, "B, Hq, Hkv, N must be >= 1");
  if (N >= kMaxN) return fail(ATTNFUSE_ERR_INVALID_ARG, "N=%d exceeds the supported maximum %d", N, kMaxN - 1);
  if (Hq % Hkv != 0) return fail(ATTNFUSE_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
  if (mode != ATTNFUSE_FUSED && mode != ATTNFUSE_PREROTATE && mode != ATTNFUSE_AUTO && mode != ATTNFUSE_SPLIT &&
      mode != ATTNFUSE_NONE)
    return fail(ATTNFUSE_ERR_INVALID_ARG, "mode %d is not fused (0), prerotate (1), auto (2), split (3) or none (4)",
                (int)mode);
  attnfuse_status_t st = check_dtype_d(d, dtype);
  if (st != ATTNFUSE_OK) return st;
  if ((st = check_base(base)) != ATTNFUSE_OK) return st;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
    return fail(ATTNFUSE_ERR_INVALID_ARG, "q, k, v and out must be 16-byte aligned");
  if (lse && !aligned(lse, 4)) return fail(ATTNFUSE_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  const long long units = (long long)B * Hq * ((N + 255) / 256);
  if (units > 0x7FFFFFFFLL) return fail(ATTNFUSE_ERR_INVALID_ARG, "problem too large: %lld work units", units);
  return ATTNFUSE_OK;
}

}  // namespace

namespace attnfuse {

void set_last_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
}

attnfuse_status_t check_fwd_call(const void* q, const void* k, const void* v, const void* out, const float* lse, int B,
                                 int Hq, int Hkv, int N, int d, double rope_base, attnfuse_mode_t mode,
                                 attnfuse_dtype_t dtype) {
  g_err[0] = '\0';
  const attnfuse_status_t st = validate_fwd(q, k, v, out, lse, B, Hq, Hkv, N, d, rope_base, mode, dtype);
  if (st != ATTNFUSE_OK) return st;
  return check_device();
}

}  // namespace attnfuse

extern "C" {

const char* attnfuse_version(void) { return "libattnfuse 0.1 (sm_103a)"; }

const char* attnfuse_status_string(attnfuse_status_t s) {
  switch (s) {
    case ATTNFUSE_OK: return "ok";
    case ATTNFUSE_ERR_INVALID_ARG: return "invalid argument";
    case ATTNFUSE_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case ATTNFUSE_ERR_CUDA: return "CUDA error";
    case ATTNFUSE_ERR_TIMEOUT: return "a kernel barrier wait timed out";
    case ATTNFUSE_ERR_NO_MEMORY: return "out of device memory";
  }
  return "unknown status";
}

const char* attnfuse_last_error(void) { return g_err; }

attnfuse_mode_t attnfuse_select_mode(int B, int Hq, int Hkv, int N, int d, attnfuse_dtype_t dtype) {
  (void)d;
  (void)dtype;
  if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || Hq % Hkv != 0) return ATTNFUSE_FUSED;
  // Measured on GB300 (bench.py --sweep, N from 1024 to 16384 at 16384 tokens, bf16 and fp16): with
  // 4:1 GQA, rotating K in a pass and Q on chip (split) is fastest at all 14 points (fused beats
  // pre-rotation only below N* = 1244 in bf16, 1347 in fp16); with MHA d = 64, fused is fastest at
  // N = 1024 and 1536, pre-rotation at 2048 (interpolated fused-vs-pre-rotate N* = 1892 in both
  // dtypes), pre-rotation and split tie at 4096 and split leads (by 0.9-1.7%) from 5500 on.
  if (Hq / Hkv >= 2) return N >= 1024 ? ATTNFUSE_SPLIT : ATTNFUSE_FUSED;
  if (N >= 4096) return ATTNFUSE_SPLIT;
  return N >= 1892 ? ATTNFUSE_PREROTATE : ATTNFUSE_FUSED;
}

size_t attnfuse_workspace_bytes(int B, int Hq, int Hkv, int N, int d, attnfuse_mode_t mode, attnfuse_dtype_t dtype) {
  return attnfuse_workspace_bytes_ex(B, Hq, Hkv, N, d, mode, dtype, nullptr);
}

size_t attnfuse_workspace_bytes_ex(int B, int Hq, int Hkv, int N, int d, attnfuse_mode_t mode, attnfuse_dtype_t dtype,
                                   const attnfuse_rope_opts_t* opts) {
  if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || (d != 64 && d != 128)) return 0;
  if (dtype != ATTNFUSE_BF16 && dtype != ATTNFUSE_FP16) return 0;
  const int Nk = (opts && opts->kv_len) ? opts->kv_len : N;
  if (Nk < N) return 0;
  if (Hq % Hkv != 0) return 0;
  if (decode_eligible(B, Hq, Hkv, N, mode)) return decode_workspace_bytes(B, Hkv, Nk, d, (Hq / Hkv) * N);
  if (mode == ATTNFUSE_AUTO) mode = attnfuse_select_mode(B, Hq, Hkv, Nk, d, dtype);
  if (mode == ATTNFUSE_SPLIT) return round_up(tensor_bytes(B, Nk, Hkv, d), 256);
  if (mode != ATTNFUSE_PREROTATE) return 0;  // FUSED, NONE
  return round_up(tensor_bytes(B, N, Hq, d), 256) + round_up(tensor_bytes(B, Nk, Hkv, d), 256);
}

attnfuse_status_t attnfuse_rope_apply(const void* x, void* y, int B, int N, int H, int d, double rope_base,
                                      attnfuse_dtype_t dtype, void* stream) {
  return attnfuse_rope_apply_ex(x, y, B, N, H, d, rope_base, dtype, nullptr, stream);
}

attnfuse_status_t attnfuse_rope_apply_ex(const void* x, void* y, int B, int N, int H, int d, double rope_base,
                                         attnfuse_dtype_t dtype, const attnfuse_rope_opts_t* opts, void* stream) {
  g_err[0] = '\0';
  if (!x || !y) return fail(ATTNFUSE_ERR_INVALID_ARG, "x and y must be non-null");
  if (B < 1 || N < 1 || H < 1) return fail(ATTNFUSE_ERR_INVALID_ARG, "B, N, H must be >= 1");
  if (N >= kMaxN) return fail(ATTNFUSE_ERR_INVALID_ARG, "N=%d exceeds the supported maximum %d", N, kMaxN - 1);
  attnfuse_status_t st = check_dtype_d(d, dtype);
  if (st != ATTNFUSE_OK) return st;
  if ((st = check_base(rope_base)) != ATTNFUSE_OK) return st;
  if (!aligned(x, 16) || !aligned(y, 16)) return fail(ATTNFUSE_ERR_INVALID_ARG, "x and y must be 16-byte aligned");
  const size_t bytes = tensor_bytes(B, N, H, d);
  const char* xs = static_cast<const char*>(x);
  const char* ys = static_cast<const char*>(y);
  if (xs != ys && xs < ys + bytes && ys < xs + bytes) return fail(ATTNFUSE_ERR_INVALID_ARG, "x and y overlap without being equal");
  Opts o;
  if ((st = resolve_opts(opts, d, N, &o)) != ATTNFUSE_OK) return st;
  if (o.Nk != N || o.kpos)
    return fail(ATTNFUSE_ERR_INVALID_ARG, "attnfuse_rope_apply_ex takes q_positions only (kv_len 0, k_positions NULL)");
  if ((st = check_device()) != ATTNFUSE_OK) return st;

  RopeApplyParams p;
  std::memset(&p, 0, sizeof p);
  p.job[0].x = x;
  p.job[0].y = y;
  p.job[0].H = H;
  p.job[0].groups = (H + kHeadsPerGroup - 1) / kHeadsPerGroup;
  p.njobs = 1;
  p.N = N;
  p.tokens = (long long)B * N;
  p.groups_total = p.job[0].groups;
  p.pos = o.qpos;
  p.pos_off = 0;
  p.rot_chunks = o.rdim / 16;
  p.interleaved = o.interleaved;
  rope_freqs_host(o.rdim, rope_base, &p.freqs);
  cudaError_t e = launch_rope_apply(p, d, dtype == ATTNFUSE_BF16, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rope_apply launch");
  return ATTNFUSE_OK;
}

attnfuse_status_t attnfuse_rope_causal_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                                           int Hq, int Hkv, int N, int d, double rope_base, attnfuse_mode_t mode,
                                           attnfuse_dtype_t dtype, void* workspace, size_t workspace_bytes,
                                           void* stream) {
  return attnfuse_rope_causal_fwd_ex(q, k, v, out, lse, B, Hq, Hkv, N, d, rope_base, mode, dtype, workspace,
                                     workspace_bytes, nullptr, stream);
}

attnfuse_status_t attnfuse_rope_causal_fwd_ex(const void* q, const void* k, const void* v, void* out, float* lse,
                                              int B, int Hq, int Hkv, int N, int d, double rope_base,
                                              attnfuse_mode_t mode, attnfuse_dtype_t dtype, void* workspace,
                                              size_t workspace_bytes, const attnfuse_rope_opts_t* opts,
                                              void* stream) {
  g_err[0] = '\0';
  attnfuse_status_t st = validate_fwd(q, k, v, out, lse, B, Hq, Hkv, N, d, rope_base, mode, dtype);
  if (st != ATTNFUSE_OK) return st;
  Opts o;
  if ((st = resolve_opts(opts, d, N, &o)) != ATTNFUSE_OK) return st;
  if (mode == ATTNFUSE_NONE && (o.rdim != d || o.interleaved || o.qpos || o.kpos))
    return fail(ATTNFUSE_ERR_INVALID_ARG, "mode none (no rotation) takes kv_len only: no rotary_dim, interleaved or positions");
  const int Nk = o.Nk;
  const bool decode = decode_eligible(B, Hq, Hkv, N, mode);
  if (mode == ATTNFUSE_AUTO && !decode) mode = attnfuse_select_mode(B, Hq, Hkv, Nk, d, dtype);
  const size_t need = attnfuse_workspace_bytes_ex(B, Hq, Hkv, N, d, mode, dtype, opts);
  if (workspace) {
    if (workspace_bytes < need)
      return fail(ATTNFUSE_ERR_INVALID_ARG, "workspace has %zu bytes, %zu needed", workspace_bytes, need);
    if (!aligned(workspace, 256)) return fail(ATTNFUSE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  }
  if ((st = check_device()) != ATTNFUSE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (decode) {
    DecodeParams dp;
    std::memset(&dp, 0, sizeof dp);
    dp.q = q;
    dp.k = k;
    dp.v = v;
    dp.out = out;
    dp.lse = lse;
    dp.B = B;
    dp.Hq = Hq;
    dp.Hkv = Hkv;
    dp.N = N;
    dp.Nk = Nk;
    dp.q_off = Nk - N;
    dp.qpos = o.qpos;
    dp.kpos = o.kpos;
    dp.rot_chunks = o.rdim / 16;
    dp.interleaved = o.interleaved;
    decode_plan(B, Hkv, Nk, d, (Hq / Hkv) * N, &dp.keys_per_split, &dp.n_splits);
    dp.warps = decode_warps(B, Hkv, d, (Hq / Hkv) * N);
    dp.scale_log2 = (float)(1.4426950408889634074 / std::sqrt((double)d));
    rope_freqs_host(o.rdim, rope_base, &dp.freqs);
    void* owned = nullptr;
    void* ws = workspace;
    if (!ws) {
      cudaError_t e = cudaMallocAsync(&owned, need, s);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(ATTNFUSE_ERR_NO_MEMORY, "cudaMallocAsync(%zu) for the decode partials failed: %s", need,
                    cudaGetErrorString(e));
      }
      ws = owned;
    }
    const size_t slots = (size_t)B * Hkv * dp.n_splits * kDecodeMaxRows;
    dp.part_o = static_cast<float*>(ws);
    dp.part_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + round_up(slots * d * sizeof(float), 256));
    DecodeMaps dm;
    if ((st = encode_bnhd(&dm.k, k, B, Nk, Hkv, d, dtype, "k", kDecodeChunk)) != ATTNFUSE_OK ||
        (st = encode_bnhd(&dm.v, v, B, Nk, Hkv, d, dtype, "v", kDecodeChunk)) != ATTNFUSE_OK) {
      if (owned) cudaFreeAsync(owned, s);
      return st;
    }
    cudaError_t e = launch_attn_decode(dm, dp, d, dtype == ATTNFUSE_BF16, s);
    if (owned) cudaFreeAsync(owned, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return ATTNFUSE_OK;
  }

  AttnParams p;
  std::memset(&p, 0, sizeof p);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.Nk = Nk;
  p.q_off = Nk - N;
  p.qpos = o.qpos;
  p.kpos = o.kpos;
  // GQA with an even group size pairs two query heads of a KV group on the same rows (equal key
  // ranges: no half-empty last step, finer units for the persistent schedule); otherwise a unit is
  // two consecutive 128-row tiles of one head.
  p.head_pairs = (Hq / Hkv) % 2 == 0 ? 1 : 0;
  p.n_qblocks = p.head_pairs ? (N + 127) / 128 : (N + 255) / 256;
  p.total_units = p.head_pairs ? B * (Hq / 2) * p.n_qblocks : B * Hq * p.n_qblocks;
  p.out = out;
  p.lse = lse;
  p.scale_log2 = (float)(1.4426950408889634074 / std::sqrt((double)d));
  p.timeout_ns = kTimeoutNs;
  p.rot_chunks = o.rdim / 16;
  p.interleaved = o.interleaved;
  rope_freqs_host(o.rdim, rope_base, &p.freqs);

  const void* qa = q;
  const void* ka = k;
  void* owned = nullptr;
  if (mode == ATTNFUSE_SPLIT) {
    // K (re-read by every query tile that needs it) is rotated once into the workspace; the
    // attention kernel rotates each query tile, which it reads once, on chip.
    void* ws = workspace;
    if (!ws) {
      cudaError_t e = cudaMallocAsync(&owned, need, s);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(ATTNFUSE_ERR_NO_MEMORY, "cudaMallocAsync(%zu) for the rotated K failed: %s", need, cudaGetErrorString(e));
      }
      ws = owned;
    }
    RopeApplyParams rp;
    std::memset(&rp, 0, sizeof rp);
    rp.job[0] = RopeJob{k, ws, Hkv, (Hkv + kHeadsPerGroup - 1) / kHeadsPerGroup};
    rp.njobs = 1;
    rp.N = Nk;
    rp.tokens = (long long)B * Nk;
    rp.groups_total = rp.job[0].groups;
    rp.pos = o.kpos;
    rp.pos_off = 0;
    rp.rot_chunks = p.rot_chunks;
    rp.interleaved = p.interleaved;
    rp.freqs = p.freqs;
    cudaError_t e = launch_rope_apply(rp, d, dtype == ATTNFUSE_BF16, s);
    if (e != cudaSuccess) {
      if (owned) cudaFreeAsync(owned, s);
      return cuda_fail(e, "rope_apply launch");
    }
    ka = ws;
    p.after_rope_pass = 1;
  } else if (mode == ATTNFUSE_PREROTATE) {
    void* ws = workspace;
    if (!ws) {
      cudaError_t e = cudaMallocAsync(&owned, need, s);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(ATTNFUSE_ERR_NO_MEMORY, "cudaMallocAsync(%zu) for the rotated Q/K failed: %s", need, cudaGetErrorString(e));
      }
      ws = owned;
    }
    void* qr = ws;
    void* kr = static_cast<char*>(ws) + round_up(tensor_bytes(B, N, Hq, d), 256);
    RopeApplyParams rp;
    std::memset(&rp, 0, sizeof rp);
    rp.rot_chunks = p.rot_chunks;
    rp.interleaved = p.interleaved;
    rp.freqs = p.freqs;
    const RopeJob jq{q, qr, Hq, (Hq + kHeadsPerGroup - 1) / kHeadsPerGroup};
    const RopeJob jk{k, kr, Hkv, (Hkv + kHeadsPerGroup - 1) / kHeadsPerGroup};
    cudaError_t e = cudaSuccess;
    if (Nk == N && !o.qpos && !o.kpos) {
      // Q and K share tokens and positions: one launch over both.
      rp.job[0] = jq;
      rp.job[1] = jk;
      rp.njobs = 2;
      rp.N = N;
      rp.tokens = (long long)B * N;
      rp.groups_total = jq.groups + jk.groups;
      e = launch_rope_apply(rp, d, dtype == ATTNFUSE_BF16, s);
    } else {
      // Queries at Nk - N + i (or q_positions), keys at j (or k_positions): one launch each.
      rp.njobs = 1;
      rp.job[0] = jq;
      rp.N = N;
      rp.tokens = (long long)B * N;
      rp.groups_total = jq.groups;
      rp.pos = o.qpos;
      rp.pos_off = Nk - N;
      e = launch_rope_apply(rp, d, dtype == ATTNFUSE_BF16, s);
      if (e == cudaSuccess) {
        rp.job[0] = jk;
        rp.N = Nk;
        rp.tokens = (long long)B * Nk;
        rp.groups_total = jk.groups;
        rp.pos = o.kpos;
        rp.pos_off = 0;
        e = launch_rope_apply(rp, d, dtype == ATTNFUSE_BF16, s);
      }
    }
    if (e != cudaSuccess) {
      if (owned) cudaFreeAsync(owned, s);
      return cuda_fail(e, "rope_apply launch");
    }
    qa = qr;
    ka = kr;
    p.after_rope_pass = 1;
  }

  AttnMaps maps;
  if ((st = encode_bnhd(&maps.q, qa, B, N, Hq, d, dtype, "q")) == ATTNFUSE_OK &&
      (st = encode_bnhd(&maps.k, ka, B, Nk, Hkv, d, dtype, "k")) == ATTNFUSE_OK &&
      (st = encode_bnhd(&maps.v, v, B, Nk, Hkv, d, dtype, "v")) == ATTNFUSE_OK) {
    const char* why = nullptr;
    cudaError_t e = launch_attn_fwd(maps, p, d, dtype == ATTNFUSE_BF16, mode == ATTNFUSE_FUSED || mode == ATTNFUSE_SPLIT,
                                    mode == ATTNFUSE_FUSED, s, &why);
    if (e != cudaSuccess) st = why ? fail(ATTNFUSE_ERR_UNSUPPORTED, "%s", why) : cuda_fail(e, "attention launch");
  }
  if (owned) cudaFreeAsync(owned, s);
  return st;
}

size_t attnfuse_bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d, attnfuse_dtype_t dtype) {
  return attnfuse_bwd_workspace_bytes_ex(B, Hq, Hkv, N, d, dtype, nullptr);
}

size_t attnfuse_bwd_workspace_bytes_ex(int B, int Hq, int Hkv, int N, int d, attnfuse_dtype_t dtype,
                                       const attnfuse_rope_opts_t* opts) {
  if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || (d != 64 && d != 128)) return 0;
  if (dtype != ATTNFUSE_BF16 && dtype != ATTNFUSE_FP16) return 0;
  const int Nk = (opts && opts->kv_len) ? opts->kv_len : N;
  if (Nk < N) return 0;
  return round_up(tensor_bytes(B, N, Hq, d), 256) + round_up(tensor_bytes(B, Nk, Hkv, d), 256) +
         round_up((size_t)B * Hq * N * sizeof(float), 256) + 256;  // + the dQ kernel's unit counter
}

attnfuse_status_t attnfuse_rope_causal_bwd(const void* q, const void* k, const void* v, const void* out,
                                           const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                                           int Hq, int Hkv, int N, int d, double rope_base, attnfuse_dtype_t dtype,
                                           void* workspace, size_t workspace_bytes, void* stream) {
  return attnfuse_rope_causal_bwd_ex(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, rope_base, dtype, workspace,
                                     workspace_bytes, nullptr, stream);
}

attnfuse_status_t attnfuse_rope_causal_bwd_ex(const void* q, const void* k, const void* v, const void* out,
                                              const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                                              int Hq, int Hkv, int N, int d, double rope_base, attnfuse_dtype_t dtype,
                                              void* workspace, size_t workspace_bytes,
                                              const attnfuse_rope_opts_t* opts, void* stream) {
  g_err[0] = '\0';
  attnfuse_status_t st = validate_fwd(q, k, v, out, lse, B, Hq, Hkv, N, d, rope_base, ATTNFUSE_FUSED, dtype);
  if (st != ATTNFUSE_OK) return st;
  Opts o;
  if ((st = resolve_opts(opts, d, N, &o)) != ATTNFUSE_OK) return st;
  const int Nk = o.Nk;
  // The half-split form over all d at positions i and j is rotated back in the kernels' epilogues;
  // any other form runs a pre-rotation pass with the negated positions over dq and dk afterwards.
  const bool plain_form = o.rdim == d && o.interleaved == 0 && !o.qpos && !o.kpos;
  if (!lse || !dout || !dq || !dk || !dv) return fail(ATTNFUSE_ERR_INVALID_ARG, "lse, dout, dq, dk and dv must be non-null");
  if (!aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16))
    return fail(ATTNFUSE_ERR_INVALID_ARG, "dout, dq, dk and dv must be 16-byte aligned");
  const size_t need = attnfuse_bwd_workspace_bytes_ex(B, Hq, Hkv, N, d, dtype, opts);
  if (workspace) {
    if (workspace_bytes < need)
      return fail(ATTNFUSE_ERR_INVALID_ARG, "workspace has %zu bytes, %zu needed", workspace_bytes, need);
    if (!aligned(workspace, 256)) return fail(ATTNFUSE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  }
  if ((st = check_device()) != ATTNFUSE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  void* owned = nullptr;
  void* ws = workspace;
  if (!ws) {
    cudaError_t e = cudaMallocAsync(&owned, need, s);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(ATTNFUSE_ERR_NO_MEMORY, "cudaMallocAsync(%zu) for the backward workspace failed: %s", need,
                  cudaGetErrorString(e));
    }
    ws = owned;
  }
  void* qr = ws;
  void* kr = static_cast<char*>(ws) + round_up(tensor_bytes(B, N, Hq, d), 256);
  float* Dv = reinterpret_cast<float*>(static_cast<char*>(kr) + round_up(tensor_bytes(B, Nk, Hkv, d), 256));
  int* unit_ctr = reinterpret_cast<int*>(reinterpret_cast<char*>(Dv) + round_up((size_t)B * Hq * N * sizeof(float), 256));

  AttnBwdParams p;
  std::memset(&p, 0, sizeof p);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.Nk = Nk;
  p.q_off = Nk - N;
  p.n_tiles = (N + 127) / 128;
  p.n_ktiles = (Nk + 127) / 128;
  p.out = out;
  p.dout = dout;
  p.lse = lse;
  p.Dvec = Dv;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.scale_log2 = (float)(1.4426950408889634074 / std::sqrt((double)d));
  p.inv_sqrt_d = (float)(1.0 / std::sqrt((double)d));
  p.unrotate = plain_form ? 1 : 0;
  p.timeout_ns = kTimeoutNs;
  p.unit_ctr = unit_ctr;
  rope_freqs_host(d, rope_base, &p.freqs);

  // One pre-rotation launch per tensor (queries at q_off + i or q_positions over N tokens, keys at j
  // or k_positions over Nk), or both tensors in one launch when they share tokens and positions.
  // neg = 0: q', k' before the kernels; 1: dq, dk rotated back after them (R(p)^T = R(-p)).
  RopeApplyParams rp;
  std::memset(&rp, 0, sizeof rp);
  rp.rot_chunks = o.rdim / 16;
  rp.interleaved = o.interleaved;
  rope_freqs_host(o.rdim, rope_base, &rp.freqs);
  auto rotate = [&](const void* xq, void* yq, const void* xk, void* yk, int neg) -> cudaError_t {
    rp.pos_neg = neg;
    const RopeJob jq{xq, yq, Hq, (Hq + kHeadsPerGroup - 1) / kHeadsPerGroup};
    const RopeJob jk{xk, yk, Hkv, (Hkv + kHeadsPerGroup - 1) / kHeadsPerGroup};
    if (Nk == N && !o.qpos && !o.kpos) {
      rp.job[0] = jq;
      rp.job[1] = jk;
      rp.njobs = 2;
      rp.N = N;
      rp.tokens = (long long)B * N;
      rp.groups_total = jq.groups + jk.groups;
      rp.pos = nullptr;
      rp.pos_off = 0;
      return launch_rope_apply(rp, d, dtype == ATTNFUSE_BF16, s);
    }
    rp.njobs = 1;
    rp.job[0] = jq;
    rp.N = N;
    rp.tokens = (long long)B * N;
    rp.groups_total = jq.groups;
    rp.pos = o.qpos;
    rp.pos_off = Nk - N;
    cudaError_t err = launch_rope_apply(rp, d, dtype == ATTNFUSE_BF16, s);
    if (err != cudaSuccess) return err;
    rp.job[0] = jk;
    rp.N = Nk;
    rp.tokens = (long long)B * Nk;
    rp.groups_total = jk.groups;
    rp.pos = o.kpos;
    rp.pos_off = 0;
    return launch_rope_apply(rp, d, dtype == ATTNFUSE_BF16, s);
  };
  cudaError_t e = rotate(q, qr, k, kr, 0);
  if (e != cudaSuccess) st = cuda_fail(e, "rope_apply launch");
  AttnBwdMaps maps;
  if (st == ATTNFUSE_OK && (st = encode_bnhd(&maps.q, qr, B, N, Hq, d, dtype, "q'")) == ATTNFUSE_OK &&
      (st = encode_bnhd(&maps.k, kr, B, Nk, Hkv, d, dtype, "k'")) == ATTNFUSE_OK &&
      (st = encode_bnhd(&maps.v, v, B, Nk, Hkv, d, dtype, "v")) == ATTNFUSE_OK &&
      (st = encode_bnhd(&maps.dout, dout, B, N, Hq, d, dtype, "dout")) == ATTNFUSE_OK &&
      (st = encode_bnhd(&maps.q64, qr, B, N, Hq, d, dtype, "q'", 64)) == ATTNFUSE_OK &&
      (st = encode_bnhd(&maps.k64, kr, B, Nk, Hkv, d, dtype, "k'", 64)) == ATTNFUSE_OK &&
      (st = encode_bnhd(&maps.v64, v, B, Nk, Hkv, d, dtype, "v", 64)) == ATTNFUSE_OK &&
      (st = encode_bnhd(&maps.dout64, dout, B, N, Hq, d, dtype, "dout", 64)) == ATTNFUSE_OK) {
    e = launch_attn_bwd(maps, p, d, dtype == ATTNFUSE_BF16, s);
    if (e != cudaSuccess) st = cuda_fail(e, "backward launch");
    if (st == ATTNFUSE_OK && !plain_form && (e = rotate(dq, dq, dk, dk, 1)) != cudaSuccess)
      st = cuda_fail(e, "rope_apply launch (rotating the gradients back)");
  }
  if (owned) cudaFreeAsync(owned, s);
  return st;
}

attnfuse_status_t attnfuse_device_status(void* stream) {
  g_err[0] = '\0';
  unsigned int v = 0;
  cudaError_t e = read_and_clear_device_status(&v, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "device status");
  unsigned int vb = 0;
  e = read_and_clear_bwd_status(&vb);
  if (e != cudaSuccess) return cuda_fail(e, "device status (backward)");
  v |= vb;
  unsigned int vd = 0;
  e = read_and_clear_decode_status(&vd);
  if (e != cudaSuccess) return cuda_fail(e, "device status (decode)");
  v |= vd;
  if (v != 0u) return fail(ATTNFUSE_ERR_TIMEOUT, "a kernel barrier wait ran out (device status 0x%x)", v);
  return ATTNFUSE_OK;
}

attnfuse_status_t attnfuse_diag_wait_timeout(uint64_t timeout_ns, void* stream) {
  g_err[0] = '\0';
  if (timeout_ns == 0 || timeout_ns > 1000000000ull) return fail(ATTNFUSE_ERR_INVALID_ARG, "timeout_ns must be in (0, 1e9]");
  attnfuse_status_t st = check_device();
  if (st != ATTNFUSE_OK) return st;
  cudaError_t e = launch_diag_wait_timeout((unsigned long long)timeout_ns, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "diag launch");
  return ATTNFUSE_OK;
}

}  // extern "C"
