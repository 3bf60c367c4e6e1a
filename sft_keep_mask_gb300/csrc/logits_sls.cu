// Scoring of logits that already exist: selected-token log-prob, entropy and
// log-sum-exp of each row of a [N, V] logit matrix, and the gradient with
// respect to the logits -- the chunked, float32 `selective_log_softmax` of
// twinkle pull request #283, section 1 ("selective_log_softmax pins one
// full-vocab copy per row"): computed in float32 from bf16 (or float32)
// logits, results in float32, nothing saved for the backward but lse and
// entropy (the softmax is recomputed from the logits).
//
// One CTA of 256 threads per row.  Each thread walks the row in 16-byte
// vectors, keeping a max-shifted online (m, s = sum 2^(z2-m),
// u = sum 2^(z2-m) (z2-m)) in log2 units; the CTA merges the 256 partials.
// The work is bound by HBM bandwidth: 2 bytes per bf16 logit read in the
// forward; read + write in the backward.
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace lmhead {
namespace {

constexpr int kSlsThreads = 256;
constexpr float kSlsLog2e = 1.4426950408889634f;
constexpr float kSlsLn2 = 0.6931471805599453f;

__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(float v) { return v; }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}
template <>
__device__ __forceinline__ float from_f32<float>(float v) {
  return v;
}

struct Online {
  float m;  // running max, log2 units
  float s;  // sum 2^(z2 - m)
  float u;  // sum 2^(z2 - m) (z2 - m)

  __device__ __forceinline__ void add_block(const float* z2, int n) {
    float bm = z2[0];
    for (int j = 1; j < n; ++j) bm = fmaxf(bm, z2[j]);
    if (bm > m) {
      if (m != -INFINITY) {
        const float sc = fast_exp2(m - bm);
        u = sc * (u + s * (m - bm));
        s *= sc;
      }
      m = bm;
    }
    for (int j = 0; j < n; ++j) {
      const float d = z2[j] - m;
      const float e = fast_exp2(d);
      s += e;
      u = fmaf(e, d, u);
    }
  }

  __device__ __forceinline__ void merge(float m2, float s2, float u2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) {
      m = m2; s = s2; u = u2;
      return;
    }
    const float M = fmaxf(m, m2);
    const float a = fast_exp2(m - M), b = fast_exp2(m2 - M);
    u = a * (u + s * (m - M)) + b * (u2 + s2 * (m2 - M));
    s = a * s + b * s2;
    m = M;
  }
};

// Loads 16 bytes of row z at element offset e as floats scaled by log2(e).
template <typename T>
__device__ __forceinline__ int load_vec_log2(const T* z, int64_t e, float* out);

template <>
__device__ __forceinline__ int load_vec_log2<__nv_bfloat16>(const __nv_bfloat16* z, int64_t e,
                                                            float* out) {
  const uint4 v = *reinterpret_cast<const uint4*>(z + e);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    out[2 * j] = __uint_as_float(w[j] << 16) * kSlsLog2e;
    out[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u) * kSlsLog2e;
  }
  return 8;
}

template <>
__device__ __forceinline__ int load_vec_log2<float>(const float* z, int64_t e, float* out) {
  const float4 v = *reinterpret_cast<const float4*>(z + e);
  out[0] = v.x * kSlsLog2e;
  out[1] = v.y * kSlsLog2e;
  out[2] = v.z * kSlsLog2e;
  out[3] = v.w * kSlsLog2e;
  return 4;
}

template <typename T>
__global__ void __launch_bounds__(kSlsThreads) sls_fwd_kernel(
    const T* __restrict__ logits, int64_t ld, bool vec_ok, const int64_t* __restrict__ targets,
    const uint8_t* __restrict__ keep, int V, int want_entropy, float* __restrict__ lp,
    float* __restrict__ ent, float* __restrict__ lse, int* status) {
  const int64_t row = blockIdx.x;
  if (keep != nullptr && keep[row] == 0) {
    if (threadIdx.x == 0) {
      lp[row] = 0.f;
      lse[row] = 0.f;
      if (ent) ent[row] = 0.f;
    }
    return;
  }
  const T* z = logits + row * ld;
  constexpr int E = 16 / sizeof(T);
  Online o{-INFINITY, 0.f, 0.f};
  int64_t scalar_from = 0;
  if (vec_ok) {
    const int64_t nvec = V / E;
    int64_t i = threadIdx.x;
    // two vectors in flight per iteration
    for (; i + kSlsThreads < nvec; i += 2 * kSlsThreads) {
      float a[E], b[E];
      load_vec_log2<T>(z, i * E, a);
      load_vec_log2<T>(z, (i + kSlsThreads) * E, b);
      o.add_block(a, E);
      o.add_block(b, E);
    }
    for (; i < nvec; i += kSlsThreads) {
      float a[E];
      load_vec_log2<T>(z, i * E, a);
      o.add_block(a, E);
    }
    scalar_from = nvec * E;
  }
  for (int64_t e = scalar_from + threadIdx.x; e < V; e += kSlsThreads) {
    const float a = to_f32(z[e]) * kSlsLog2e;
    o.add_block(&a, 1);
  }
  // merge the 256 partials
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, o.m, off);
    const float s2 = __shfl_xor_sync(0xffffffffu, o.s, off);
    const float u2 = __shfl_xor_sync(0xffffffffu, o.u, off);
    o.merge(m2, s2, u2);
  }
  __shared__ float sm[kSlsThreads / 32][3];
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    sm[w][0] = o.m;
    sm[w][1] = o.s;
    sm[w][2] = o.u;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    Online t{-INFINITY, 0.f, 0.f};
    for (int j = 0; j < kSlsThreads / 32; ++j) t.merge(sm[j][0], sm[j][1], sm[j][2]);
    int64_t y = targets[row];
    if (y < 0 || y >= V) {
      if (status != nullptr) atomicCAS(status, 0, kStatusTarget);
      y = 0;
    }
    const float logS = logf(t.s);
    const float l_row = t.m * kSlsLn2 + logS;
    lse[row] = l_row;
    lp[row] = to_f32(z[y]) - l_row;
    if (want_entropy) ent[row] = logS - (t.u * kSlsLn2) / t.s;
  }
}

template <typename T>
__global__ void __launch_bounds__(kSlsThreads) sls_bwd_kernel(
    const T* __restrict__ logits, int64_t ld, bool vec_ok, const int64_t* __restrict__ targets,
    const uint8_t* __restrict__ keep, int V, const float* __restrict__ lse,
    const float* __restrict__ ent, const float* __restrict__ g_lp,
    const float* __restrict__ g_ent, T* __restrict__ dz, int64_t ld_out, int* status) {
  const int64_t row = blockIdx.x;
  const T* z = logits + row * ld;
  T* g = dz + row * ld_out;
  constexpr int E = 16 / sizeof(T);
  const bool kept = keep == nullptr || keep[row] != 0;
  float lse2 = 0.f, ca = 0.f, cb = 0.f, glp = 0.f;
  int64_t y = -1;
  if (kept) {
    lse2 = lse[row] * kSlsLog2e;
    glp = g_lp[row];
    if (g_ent != nullptr) {
      ca = g_ent[row] * kSlsLn2;
      cb = glp + g_ent[row] * ent[row];
    } else {
      cb = glp;
    }
    y = targets[row];
    if (y < 0 || y >= V) {
      if (threadIdx.x == 0 && status != nullptr) atomicCAS(status, 0, kStatusTarget);
      y = 0;
    }
  }
  auto grad = [&](float zv, int64_t e) -> float {
    if (!kept) return 0.f;
    const float d = fmaf(zv, kSlsLog2e, -lse2);
    const float p = fast_exp2(d);
    float r = -p * fmaf(ca, d, cb);
    if (e == y) r += glp;
    return r;
  };
  int64_t scalar_from = 0;
  if (vec_ok) {
    const int64_t nvec = V / E;
    for (int64_t i = threadIdx.x; i < nvec; i += kSlsThreads) {
      const int64_t e0 = i * E;
      if constexpr (sizeof(T) == 2) {
        const uint4 v = *reinterpret_cast<const uint4*>(z + e0);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          o[j] = pack_bf16x2(grad(__uint_as_float(w[j] << 16), e0 + 2 * j),
                             grad(__uint_as_float(w[j] & 0xFFFF0000u), e0 + 2 * j + 1));
        *reinterpret_cast<uint4*>(g + e0) = make_uint4(o[0], o[1], o[2], o[3]);
      } else {
        const float4 v = *reinterpret_cast<const float4*>(z + e0);
        *reinterpret_cast<float4*>(g + e0) =
            make_float4(grad(v.x, e0), grad(v.y, e0 + 1), grad(v.z, e0 + 2), grad(v.w, e0 + 3));
      }
    }
    scalar_from = nvec * E;
  }
  for (int64_t e = scalar_from + threadIdx.x; e < V; e += kSlsThreads)
    g[e] = from_f32<T>(grad(to_f32(z[e]), e));
}

template <typename T>
bool vec_aligned(const void* p, int64_t ld) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0 && ((ld * sizeof(T)) & 15) == 0;
}

}  // namespace

cudaError_t launch_sls_fwd(const void* logits, int dtype, int64_t ld, const int64_t* targets,
                           const uint8_t* keep, int64_t N, int V, int want_entropy, float* lp,
                           float* ent, float* lse, int* status, cudaStream_t s) {
  if (dtype == 0) {
    const bool v = vec_aligned<__nv_bfloat16>(logits, ld);
    sls_fwd_kernel<__nv_bfloat16><<<static_cast<unsigned>(N), kSlsThreads, 0, s>>>(
        static_cast<const __nv_bfloat16*>(logits), ld, v, targets, keep, V, want_entropy, lp,
        ent, lse, status);
  } else {
    const bool v = vec_aligned<float>(logits, ld);
    sls_fwd_kernel<float><<<static_cast<unsigned>(N), kSlsThreads, 0, s>>>(
        static_cast<const float*>(logits), ld, v, targets, keep, V, want_entropy, lp, ent, lse,
        status);
  }
  return cudaGetLastError();
}

cudaError_t launch_sls_bwd(const void* logits, int dtype, int64_t ld, const int64_t* targets,
                           const uint8_t* keep, int64_t N, int V, const float* lse,
                           const float* ent, const float* g_lp, const float* g_ent, void* dz,
                           int64_t ld_out, int* status, cudaStream_t s) {
  if (dtype == 0) {
    const bool v = vec_aligned<__nv_bfloat16>(logits, ld) && vec_aligned<__nv_bfloat16>(dz, ld_out);
    sls_bwd_kernel<__nv_bfloat16><<<static_cast<unsigned>(N), kSlsThreads, 0, s>>>(
        static_cast<const __nv_bfloat16*>(logits), ld, v, targets, keep, V, lse, ent, g_lp, g_ent,
        static_cast<__nv_bfloat16*>(dz), ld_out, status);
  } else {
    const bool v = vec_aligned<float>(logits, ld) && vec_aligned<float>(dz, ld_out);
    sls_bwd_kernel<float><<<static_cast<unsigned>(N), kSlsThreads, 0, s>>>(
        static_cast<const float*>(logits), ld, v, targets, keep, V, lse, ent, g_lp, g_ent,
        static_cast<float*>(dz), ld_out, status);
  }
  return cudaGetLastError();
}

}  // namespace lmhead
