// mk_noalloc.cu -- grouped-query decode attention that allocates no device
// memory: mk_attention_noalloc().
//
// Some callers cannot allocate GPU memory themselves: a serving engine that
// owns and budgets every byte of device memory through its own allocator (so
// a library may not take memory behind its back), or a latency-critical
// decode loop where a cudaMalloc and the synchronisation it implies are not
// acceptable.  They hand this entry point their own query, KV-cache and
// output buffers; the only scratch it needs -- the split-KV chunk partials --
// lives in a fixed, file-scope device array of this library.
//
// The computation is the megakernel's attention step (chunked over the KV
// positions 0..p_b, chunk partials {m, l, o} merged by log-sum-exp), run as
// two ordinary launches: one block per (chunk, KV group, sequence), then one
// block per (KV group, sequence) for the merge.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "mk.h"

namespace {

// 4 MiB of fp32 partials, held by every GPU that loads the library.
constexpr size_t kScratchFloats = size_t(1) << 20;
static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

// Host code cannot use g_noalloc_scratch as an address (it names a host-side
// stand-in); the device address is resolved once per device.
constexpr int kMaxDevices = 64;
std::mutex g_mutex;
float *g_scratch_ptr[kMaxDevices] = {};

int scratch_for_current_device(float **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return MK_ERR_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return MK_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return MK_ERR_CUDA;
    }
    g_scratch_ptr[dev] = static_cast<float *>(p);
  }
  *out = g_scratch_ptr[dev];
  return MK_OK;
}

__device__ __forceinline__ float bf(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// positions [p0, p1) of chunk c of nch over 0..pos (equal lengths, a multiple of 16)
__device__ __forceinline__ void chunk_range(int pos, int nch, int c, int &p0, int &p1) {
  const int sb = (((pos + 1) + nch - 1) / nch + 15) & ~15;
  p0 = c * sb;
  p1 = min(p0 + sb, pos + 1);
  if (p1 < p0) p1 = p0;
}

// One chunk of one KV group of one sequence: partial {m[qpg], l[qpg], o[qpg][d]}.
// 128 threads.  Scores: a warp reads DD/8 lanes' 16 bytes of each of
// 256/DD consecutive key rows at a time (whole rows, contiguous), every lane
// dots its 8 dimensions with every head's query and a butterfly over the
// row's lanes finishes each score.  Values: warp w takes rows w, w + 4, ...,
// each lane DD/32 consecutive dimensions of a row (one contiguous row per
// warp step), all heads at once; the four warps' sums meet in shared memory.
template <int DD>
__global__ void noalloc_attn_partial(const float *q, const uint16_t *kc, const uint16_t *vc,
                                     const int32_t *positions, float *part, int nq, int nkv,
                                     int max_ctx, int nch, int ch, float scale) {
  constexpr int LPP = DD / 8, RPS = 32 / LPP, DPL = DD / 32, MAXQ = 8;
  extern __shared__ float sm[];
  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int qpg = nq / nkv, PS = 2 * qpg + qpg * DD;
  float *qs = sm, *s = qs + qpg * DD, *po = s + qpg * ch;  // po: [4][qpg][DD]
  float *dst = part + (((size_t)b * nkv + g) * nch + c) * PS;
  const int pos = positions[b];
  int p0 = 0, p1 = 0;
  if (pos >= 0 && pos < max_ctx) chunk_range(pos, nch, c, p0, p1);
  const int n = p1 - p0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < qpg * DD; i += blockDim.x)
    qs[i] = q[((size_t)b * nq + (size_t)g * qpg) * DD + i] * scale;
  __syncthreads();
  const size_t base = (((size_t)b * nkv + g) * max_ctx + p0) * DD;
  const int part8 = (lane % LPP) * 8;
  for (int j0 = warp * RPS; j0 < n; j0 += 4 * RPS) {
    const int j = j0 + lane / LPP;
    float k8[8];
    if (j < n) {
      const uint4 w = *reinterpret_cast<const uint4 *>(kc + base + (size_t)j * DD + part8);
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        k8[2 * t] = __uint_as_float(u[t] << 16);
        k8[2 * t + 1] = __uint_as_float(u[t] & 0xFFFF0000u);
      }
    } else {
#pragma unroll
      for (int t = 0; t < 8; ++t) k8[t] = 0.f;
    }
    for (int h = 0; h < qpg; ++h) {
      float a = 0.f;
#pragma unroll
      for (int t = 0; t < 8; ++t) a = fmaf(qs[h * DD + part8 + t], k8[t], a);
#pragma unroll
      for (int o = LPP / 2; o; o >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
      if (j < n && lane % LPP == 0) s[h * ch + j] = a;
    }
  }
  __syncthreads();
  for (int h = warp; h < qpg; h += 4) {
    float m = -INFINITY;
    for (int j = lane; j < n; j += 32) m = fmaxf(m, s[h * ch + j]);
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    float l = 0.f;
    for (int j = lane; j < n; j += 32) {
      const float p = __expf(s[h * ch + j] - m);
      s[h * ch + j] = p;
      l += p;
    }
    for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
    if (lane == 0) {
      dst[h] = m;
      dst[qpg + h] = l;
    }
  }
  __syncthreads();
  float acc[MAXQ][DPL];
#pragma unroll
  for (int h = 0; h < MAXQ; ++h)
#pragma unroll
    for (int k = 0; k < DPL; ++k) acc[h][k] = 0.f;
  for (int j = warp; j < n; j += 4) {
    const uint16_t *vr = vc + base + (size_t)j * DD + lane * DPL;
    float v[DPL];
#pragma unroll
    for (int k = 0; k < DPL; k += 2) {
      const uint32_t w = *reinterpret_cast<const uint32_t *>(vr + k);
      v[k] = __uint_as_float(w << 16);
      v[k + 1] = __uint_as_float(w & 0xFFFF0000u);
    }
#pragma unroll
    for (int h = 0; h < MAXQ; ++h)
      if (h < qpg) {
        const float p = s[h * ch + j];
#pragma unroll
        for (int k = 0; k < DPL; ++k) acc[h][k] = fmaf(p, v[k], acc[h][k]);
      }
  }
#pragma unroll
  for (int h = 0; h < MAXQ; ++h)
    if (h < qpg)
#pragma unroll
      for (int k = 0; k < DPL; ++k) po[((size_t)warp * qpg + h) * DD + lane * DPL + k] = acc[h][k];
  __syncthreads();
  for (int i = tid; i < qpg * DD; i += blockDim.x)
    dst[2 * qpg + i] = (po[i] + po[qpg * DD + i]) + (po[2 * qpg * DD + i] + po[3 * qpg * DD + i]);
}

// Log-sum-exp merge of a group's chunk partials into out[b][(g*qpg + h)*d + k];
// a sequence whose position is out of range gets NaN.
__global__ void noalloc_attn_merge(const float *part, const int32_t *positions, float *out,
                                   int nq, int nkv, int d, int max_ctx, int nch) {
  const int g = blockIdx.x, b = blockIdx.y;
  const int qpg = nq / nkv, PS = 2 * qpg + qpg * d;
  const float *pb = part + ((size_t)b * nkv + g) * nch * PS;
  const int pos = positions[b];
  const bool ok = pos >= 0 && pos < max_ctx;
  for (int i = threadIdx.x; i < qpg * d; i += blockDim.x) {
    const int h = i / d, k = i % d;
    float M = -INFINITY, den = 0.f, num = 0.f;
    for (int c = 0; c < nch; ++c) {
      const float mc = pb[(size_t)c * PS + h];
      if (mc == -INFINITY) continue;
      const float Mn = fmaxf(M, mc);
      const float a = __expf(M - Mn), w = __expf(mc - Mn);
      den = den * a + w * pb[(size_t)c * PS + qpg + h];
      num = num * a + w * pb[(size_t)c * PS + 2 * qpg + h * d + k];
      M = Mn;
    }
    out[(size_t)b * nq * d + ((size_t)g * qpg + h) * d + k] = ok ? num / den : __int_as_float(0x7FC00000);
  }
}

}  // namespace

extern "C" MK_API int mk_attention_noalloc(const float *q, const void *k_cache,
                                           const void *v_cache, const int32_t *positions,
                                           float *out, int32_t batch, int32_t n_q_heads,
                                           int32_t n_kv_heads, int32_t head_dim, int32_t max_ctx,
                                           void *stream) {
  if (!q || !k_cache || !v_cache || !positions || !out) return MK_ERR_ARG;
  if (batch < 1 || n_kv_heads < 1 || n_q_heads < 1 || n_q_heads % n_kv_heads ||
      n_q_heads / n_kv_heads > 8 || (head_dim != 64 && head_dim != 128) || max_ctx < 16 ||
      max_ctx % 16)
    return MK_ERR_ARG;
  // chunk length: a power of two in 64..256, about max_ctx / 16
  int ch = 64;
  while (ch < 256 && ch * 16 < max_ctx) ch *= 2;
  const int nch = (max_ctx + ch - 1) / ch;
  const int qpg = n_q_heads / n_kv_heads;
  const size_t need = (size_t)batch * n_kv_heads * nch * (2 * qpg + qpg * head_dim);
  if (need > kScratchFloats) return MK_ERR_ARG;  // larger than the fixed scratch
  // An error left pending by the caller's own earlier work is reported as
  // MK_ERR_CUDA and left in place for the caller (peek, not get); each
  // launch below is checked on its own, so a rejected partial launch returns
  // before the merge is queued.
  if (cudaPeekAtLastError() != cudaSuccess) return MK_ERR_CUDA;
  float *scratch = nullptr;
  int rc = scratch_for_current_device(&scratch);
  if (rc != MK_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t smem = (size_t)(qpg * head_dim + qpg * ch + 4 * qpg * head_dim) * sizeof(float);
  const float scale = (float)(1.0 / sqrt((double)head_dim));
  const uint16_t *kc = static_cast<const uint16_t *>(k_cache);
  const uint16_t *vc = static_cast<const uint16_t *>(v_cache);
  if (head_dim == 64)
    noalloc_attn_partial<64><<<dim3(nch, n_kv_heads, batch), 128, smem, s>>>(
        q, kc, vc, positions, scratch, n_q_heads, n_kv_heads, max_ctx, nch, ch, scale);
  else
    noalloc_attn_partial<128><<<dim3(nch, n_kv_heads, batch), 128, smem, s>>>(
        q, kc, vc, positions, scratch, n_q_heads, n_kv_heads, max_ctx, nch, ch, scale);
  if (cudaGetLastError() != cudaSuccess) return MK_ERR_LAUNCH;
  noalloc_attn_merge<<<dim3(n_kv_heads, batch), 128, 0, s>>>(
      scratch, positions, out, n_q_heads, n_kv_heads, head_dim, max_ctx, nch);
  if (cudaGetLastError() != cudaSuccess) return MK_ERR_LAUNCH;
  return MK_OK;
}
