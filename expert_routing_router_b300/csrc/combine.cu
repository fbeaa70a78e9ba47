// combine.cu -- weighted un-permute + sum (combine) and the bias update.
//
// Ultralytics glossary "Expert Parallelism", section "How tokens move between GPUs",
// step 4: expert outputs return to each token's home, are weighted by the router
// scores and summed.  Section "Load balancing and capacity": a token that skipped
// its experts passes through the residual connection unchanged; after each step
// the selection bias of overloaded experts is lowered and that of underloaded
// experts raised.
//
// K5 gathers (rather than scatters) so that every output row is written exactly
// once and the sum order is fixed: acc = residual; acc += yshared; acc += w_j*y_j
// for j = 0..k-1 (kept choices only), fp32, one rounding to the output type.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int TC = 256;

template <typename T>
struct Vec;  // 16 bytes of T, widened to fp32
template <>
struct Vec<float> {
  static constexpr int n = 4;
  __device__ static void load(const void* p, float* f) {
    const uint4 v = *static_cast<const uint4*>(p);
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ static void store(void* p, const float* f) {
    *static_cast<uint4*>(p) =
        make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                   __float_as_uint(f[3]));
  }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int n = 8;
  __device__ static void load(const void* p, float* f) {
    const uint4 v = *static_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static void store(void* p, const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *static_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <typename T>
__global__ void __launch_bounds__(TC)
combine_kernel(const uint4* __restrict__ yperm, const int32_t* __restrict__ slot_of,
               const float* __restrict__ topk_w, const uint4* __restrict__ residual,
               const uint4* __restrict__ yshared, uint4* __restrict__ out, int N, int k, int nvec) {
  constexpr int L = Vec<T>::n;
  for (int t = blockIdx.x; t < N; t += gridDim.x) {
    int slots[kMaxTopK];
    float w[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      slots[j] = (j < k) ? slot_of[(int64_t)t * k + j] : -1;
      w[j] = (j < k) ? topk_w[(int64_t)t * k + j] : 0.0f;
    }
    for (int v = threadIdx.x; v < nvec; v += TC) {
      // issue every load of this vector position before any arithmetic
      uint4 raw[kMaxTopK];
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j)
        if (slots[j] >= 0) raw[j] = ld_stream_u4(yperm + (int64_t)slots[j] * nvec + v);
      uint4 rres = make_uint4(0, 0, 0, 0), rsh = make_uint4(0, 0, 0, 0);
      if (residual) rres = ld_stream_u4(residual + (int64_t)t * nvec + v);
      if (yshared) rsh = ld_stream_u4(yshared + (int64_t)t * nvec + v);
      float acc[L], tmp[L];
      if (residual) {
        Vec<T>::load(&rres, acc);
      } else {
#pragma unroll
        for (int i = 0; i < L; ++i) acc[i] = 0.0f;
      }
      if (yshared) {
        Vec<T>::load(&rsh, tmp);
#pragma unroll
        for (int i = 0; i < L; ++i) acc[i] += tmp[i];
      }
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {
        if (slots[j] >= 0) {
          Vec<T>::load(&raw[j], tmp);
#pragma unroll
          for (int i = 0; i < L; ++i) acc[i] = fmaf(w[j], tmp[i], acc[i]);
        }
      }
      Vec<T>::store(out + (int64_t)t * nvec + v, acc);
    }
  }
}

// top-1 / top-2 layers with short rows (nvec <= TC): TC / nvec tokens per CTA pass, one
// 16-byte vector per thread, and each token's two slots and weights loaded one pass
// ahead, so the row loads of a pass wait on no index load.  Same sum order as above.
template <typename T>
__global__ void __launch_bounds__(TC)
combine_k2_kernel(const uint4* __restrict__ yperm, const int32_t* __restrict__ slot_of,
                  const float* __restrict__ topk_w, const uint4* __restrict__ residual,
                  const uint4* __restrict__ yshared, uint4* __restrict__ out, int N, int k,
                  int nvec) {
  constexpr int L = Vec<T>::n;
  const int tpp = TC / nvec;              // tokens per pass
  const int sub = threadIdx.x / nvec;     // this thread's token within the pass
  const int v = threadIdx.x - sub * nvec;
  if (sub >= tpp) return;
  const int step = gridDim.x * tpp;
  int t = blockIdx.x * tpp + sub;
  int s0 = -1, s1 = -1;
  float w0 = 0.0f, w1 = 0.0f;
  if (t < N) {
    s0 = slot_of[(int64_t)t * k];
    w0 = topk_w[(int64_t)t * k];
    if (k > 1) {
      s1 = slot_of[(int64_t)t * k + 1];
      w1 = topk_w[(int64_t)t * k + 1];
    }
  }
  for (; t < N; t += step) {
    const int tn = t + step;
    int n0 = -1, n1 = -1;
    float nw0 = 0.0f, nw1 = 0.0f;
    if (tn < N) {
      n0 = slot_of[(int64_t)tn * k];
      nw0 = topk_w[(int64_t)tn * k];
      if (k > 1) {
        n1 = slot_of[(int64_t)tn * k + 1];
        nw1 = topk_w[(int64_t)tn * k + 1];
      }
    }
    uint4 r0 = make_uint4(0, 0, 0, 0), r1 = r0, rres = r0, rsh = r0;
    if (s0 >= 0) r0 = ld_stream_u4(yperm + (int64_t)s0 * nvec + v);
    if (s1 >= 0) r1 = ld_stream_u4(yperm + (int64_t)s1 * nvec + v);
    if (residual) rres = ld_stream_u4(residual + (int64_t)t * nvec + v);
    if (yshared) rsh = ld_stream_u4(yshared + (int64_t)t * nvec + v);
    float acc[L], tmp[L];
    if (residual) {
      Vec<T>::load(&rres, acc);
    } else {
#pragma unroll
      for (int i = 0; i < L; ++i) acc[i] = 0.0f;
    }
    if (yshared) {
      Vec<T>::load(&rsh, tmp);
#pragma unroll
      for (int i = 0; i < L; ++i) acc[i] += tmp[i];
    }
    if (s0 >= 0) {
      Vec<T>::load(&r0, tmp);
#pragma unroll
      for (int i = 0; i < L; ++i) acc[i] = fmaf(w0, tmp[i], acc[i]);
    }
    if (s1 >= 0) {
      Vec<T>::load(&r1, tmp);
#pragma unroll
      for (int i = 0; i < L; ++i) acc[i] = fmaf(w1, tmp[i], acc[i]);
    }
    Vec<T>::store(out + (int64_t)t * nvec + v, acc);
    s0 = n0;
    s1 = n1;
    w0 = nw0;
    w1 = nw1;
  }
}

__global__ void bias_update_kernel(const int32_t* __restrict__ counts, float* __restrict__ bias,
                                   int E, int64_t mean_num, float step) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const int64_t lhs = (int64_t)counts[e] * E;
  if (lhs > mean_num) {
    bias[e] = __fsub_rn(bias[e], step);
  } else if (lhs < mean_num) {
    bias[e] = __fadd_rn(bias[e], step);
  }
}

}  // namespace

cudaError_t launch_combine(const Cfg& c, const void* yperm, const int32_t* slot_of,
                           const float* topk_w, const void* residual, const void* yshared,
                           void* out, cudaStream_t s) {
  const int nvec = (int)((int64_t)c.d * c.act_bytes / 16);
  int grid = num_sms() * 8;
  if (grid > c.N) grid = c.N;
  const uint4* yp = static_cast<const uint4*>(yperm);
  const uint4* rs = static_cast<const uint4*>(residual);
  const uint4* ys = static_cast<const uint4*>(yshared);
  uint4* o = static_cast<uint4*>(out);
  if (c.k <= 2 && nvec <= TC) {
    const int tpp = TC / nvec;
    int g2 = num_sms() * 8;
    if ((int64_t)g2 * tpp > c.N) g2 = (c.N + tpp - 1) / tpp;
    if (c.act == MOE_DTYPE_F32)
      combine_k2_kernel<float><<<g2, TC, 0, s>>>(yp, slot_of, topk_w, rs, ys, o, c.N, c.k, nvec);
    else
      combine_k2_kernel<__nv_bfloat16><<<g2, TC, 0, s>>>(yp, slot_of, topk_w, rs, ys, o, c.N,
                                                         c.k, nvec);
  } else if (c.act == MOE_DTYPE_F32) {
    combine_kernel<float><<<grid, TC, 0, s>>>(yp, slot_of, topk_w, rs, ys, o, c.N, c.k, nvec);
  } else {
    combine_kernel<__nv_bfloat16><<<grid, TC, 0, s>>>(yp, slot_of, topk_w, rs, ys, o, c.N, c.k,
                                                       nvec);
  }
  return cudaGetLastError();
}

cudaError_t launch_bias_update(const Cfg& c, const int32_t* expert_counts, float* sel_bias,
                               float step, cudaStream_t s) {
  bias_update_kernel<<<(c.E + 255) / 256, 256, 0, s>>>(expert_counts, sel_bias, c.E, c.A, step);
  return cudaGetLastError();
}

}  // namespace moe
