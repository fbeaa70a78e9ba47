// backward.cu -- the layer's backward pass outside the expert GEMMs.
//
// The forward path (Ultralytics glossary "Expert Parallelism", section "How tokens
// move between GPUs", steps 1-4; section "Load balancing and capacity") for a fixed
// selection: the top-k choice, the capacity drops and the group limit are piecewise
// constant and pass no gradient, and the selection-only bias has none (the sign rule
// moves it).  With dout = dL/dout:
//   combine    dyperm[slot(t,j)] = w[t,j] * dout[t] (kept j);  dw[t,j] = dout[t] . y_j
//   router     logit gradient from dw (softmax / sigmoid, with and without
//              renormalisation over the k selected); dx_router = dl . Wr,
//              dWr = dl^T x, db = sum_t dl
//   dispatch   dx[t] = dout[t] + dx_shared[t] + dx_router[t] + sum_{j kept} dxperm[slot]
// Kernels (HBM- or latency-bound; fp32 accumulation, one rounding per output):
//   combine_bwd_kernel       one CTA per token: dout read once, k yperm rows read, k
//                            dyperm rows written, k dot products by block reduction
//   route_bwd_kernel         one warp per token: logits row in registers, dl row written
//   router_dx_kernel         one CTA per token: dx_router[t] = sum_e dl[t,e] Wr[e]
//                            (experts with dl = 0 skipped: k of E for renormalised or
//                            sigmoid routing)
//   router_dw_kernel         dWr and db: 8-expert x 256-column slices over all tokens,
//                            skipping the tokens whose gradient is zero there (fp32
//                            layers and small batches; bf16 layers from 128 tokens use
//                            the tensor-core GEMM of router_bwd_tc.cu)
//   dispatch_bwd_kernel      one CTA per token: the gather-sum above
#include "moe_internal.cuh"
#include "sigmoid_fixed.cuh"

namespace moe {
namespace {

constexpr int TB = 256;

template <typename T>
struct V8;  // 8 activations <-> 8 floats (one 16-byte bf16 vector / two fp32 vectors)
template <>
struct V8<__nv_bfloat16> {
  __device__ static void load(const void* row, int u, float* f) {
    const uint4 v = ld_stream_u4(static_cast<const uint4*>(row) + u);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static void store(void* row, int u, const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    static_cast<uint4*>(row)[u] = make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <>
struct V8<float> {
  __device__ static void load(const void* row, int u, float* f) {
    const uint4 a = ld_stream_u4(static_cast<const uint4*>(row) + 2 * u);
    const uint4 b = ld_stream_u4(static_cast<const uint4*>(row) + 2 * u + 1);
    f[0] = __uint_as_float(a.x); f[1] = __uint_as_float(a.y);
    f[2] = __uint_as_float(a.z); f[3] = __uint_as_float(a.w);
    f[4] = __uint_as_float(b.x); f[5] = __uint_as_float(b.y);
    f[6] = __uint_as_float(b.z); f[7] = __uint_as_float(b.w);
  }
  __device__ static void store(void* row, int u, const float* f) {
    uint4* p = static_cast<uint4*>(row) + 2 * u;
    p[0] = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
    p[1] = make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]),
                      __float_as_uint(f[7]));
  }
};

template <typename T>
__global__ void __launch_bounds__(TB)
combine_bwd_kernel(const T* __restrict__ dout, const T* __restrict__ yperm,
                   const int32_t* __restrict__ slot_of, const float* __restrict__ topk_w,
                   T* __restrict__ dyperm, float* __restrict__ dtopk_w, int N, int k, int d) {
  __shared__ float red[TB / 32][kMaxTopK];
  const int units = d / 8;
  for (int t = blockIdx.x; t < N; t += gridDim.x) {
    int slots[kMaxTopK];
    float w[kMaxTopK], dot[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      slots[j] = (j < k) ? slot_of[(int64_t)t * k + j] : -1;
      w[j] = (j < k) ? topk_w[(int64_t)t * k + j] : 0.0f;
      dot[j] = 0.0f;
    }
    const T* grow = dout + (int64_t)t * d;
    for (int u = threadIdx.x; u < units; u += TB) {
      // every load of this vector position first (k expert rows and dout), then math
      float g[8], y[kMaxTopK][8], o[8];
      V8<T>::load(grow, u, g);
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j)
        if (slots[j] >= 0) V8<T>::load(yperm + (int64_t)slots[j] * d, u, y[j]);
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {
        if (slots[j] < 0) continue;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          dot[j] = fmaf(g[i], y[j][i], dot[j]);
          o[i] = w[j] * g[i];
        }
        V8<T>::store(dyperm + (int64_t)slots[j] * d, u, o);
      }
    }
    // block sums of the k dot products, fixed order
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      float v = dot[j];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) red[warp][j] = v;
    }
    __syncthreads();
    if (threadIdx.x < k) {
      const int j = threadIdx.x;
      float v = 0.0f;
      for (int wp = 0; wp < TB / 32; ++wp) v += red[wp][j];
      dtopk_w[(int64_t)t * k + j] = slots[j] >= 0 ? v : 0.0f;
    }
    __syncthreads();
  }
}

// One warp per token.  Experts of the row live in registers (E <= 256: 8 per lane).
__global__ void __launch_bounds__(TB)
route_bwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ topk_idx,
                 const float* __restrict__ dtopk_w, float* __restrict__ dlogits, int N, int E,
                 int k, int score_fn, int normalize) {
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (TB / 32);
  for (int t = blockIdx.x * (TB / 32) + (threadIdx.x >> 5); t < N; t += warps) {
    const float* l = logits + (int64_t)t * E;
    float* o = dlogits + (int64_t)t * E;
    // the k selected experts, their gradients and scores (every lane holds all k)
    int id[kMaxTopK];
    float g[kMaxTopK], sv[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      id[j] = j < k ? topk_idx[(int64_t)t * k + j] : 0;
      g[j] = j < k ? dtopk_w[(int64_t)t * k + j] : 0.0f;
      sv[j] = 0.0f;
    }
    if (score_fn == MOE_SCORE_SIGMOID) {
      float ssum = 0.0f, wdw = 0.0f;
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j)
        if (j < k) {
          sv[j] = sigmoid_fixed(l[id[j]]);  // the forward's s_j, bit for bit
          ssum += sv[j];
        }
      if (normalize) {
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j)
          if (j < k) wdw = fmaf(sv[j] / ssum, g[j], wdw);
      }
      for (int e = lane; e < E; e += 32) o[e] = 0.0f;
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j)
          if (j < k) {
            const float dsig = sv[j] * (1.0f - sv[j]);
            o[id[j]] = normalize ? dsig * (g[j] - wdw) / ssum : dsig * g[j];
          }
      }
    } else {
      float m = -INFINITY;
      for (int e = lane; e < E; e += 32) m = fmaxf(m, l[e]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      float p[kMaxTopK];
      if (normalize) {
        float zs = 0.0f, wdw = 0.0f;
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
          p[j] = j < k ? expf(l[id[j]] - m) : 0.0f;
          zs += p[j];
        }
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) wdw = fmaf(p[j] / zs, g[j], wdw);
        for (int e = lane; e < E; e += 32) o[e] = 0.0f;
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int j = 0; j < kMaxTopK; ++j)
            if (j < k) o[id[j]] = p[j] / zs * (g[j] - wdw);
        }
      } else {
        float z = 0.0f;
        for (int e = lane; e < E; e += 32) z += expf(l[e] - m);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        float wdw = 0.0f;
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
          p[j] = j < k ? expf(l[id[j]] - m) / z : 0.0f;
          wdw = fmaf(p[j], g[j], wdw);
        }
        for (int e = lane; e < E; e += 32) {
          float v = -expf(l[e] - m) / z * wdw;
#pragma unroll
          for (int j = 0; j < kMaxTopK; ++j)
            if (j < k && id[j] == e) v = fmaf(p[j], g[j], v);
          o[e] = v;
        }
      }
    }
    __syncwarp();
  }
}

// dx_router[t, :] = sum_e dl[t, e] Wr[e, :], e ascending over the experts with dl != 0
// (k of E for renormalised or sigmoid routing): warp 0 compacts the row's nonzero
// (e, dl) pairs into shared memory in ascending order, then every thread sums its
// float4 columns over that list.
__global__ void __launch_bounds__(TB)
router_dx_kernel(const float* __restrict__ dl, const float* __restrict__ Wr,
                 float* __restrict__ dx_router, int N, int E, int d) {
  __shared__ int ids[kMaxExperts];
  __shared__ float vals[kMaxExperts];
  __shared__ int count;
  const int v4 = d / 4;
  for (int t = blockIdx.x; t < N; t += gridDim.x) {
    if (threadIdx.x < 32) {
      int n = 0;
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + threadIdx.x;
        const float v = e < E ? dl[(int64_t)t * E + e] : 0.0f;
        const unsigned nz = __ballot_sync(0xffffffffu, v != 0.0f);
        if (v != 0.0f) {
          const int pos = n + __popc(nz & ((1u << threadIdx.x) - 1u));
          ids[pos] = e;
          vals[pos] = v;
        }
        n += __popc(nz);
      }
      if (threadIdx.x == 0) count = n;
    }
    __syncthreads();
    const int n = count;
    for (int c = threadIdx.x; c < v4; c += TB) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int i = 0; i < n; ++i) {
        const float sv = vals[i];
        const float4 w = reinterpret_cast<const float4*>(Wr + (int64_t)ids[i] * d)[c];
        acc.x = fmaf(sv, w.x, acc.x);
        acc.y = fmaf(sv, w.y, acc.y);
        acc.z = fmaf(sv, w.z, acc.z);
        acc.w = fmaf(sv, w.w, acc.w);
      }
      reinterpret_cast<float4*>(dx_router + (int64_t)t * d)[c] = acc;
    }
    __syncthreads();
  }
}

// dWr [E, d] = sum_t dl[t, e] x[t, :] and db [E] = sum_t dl[t, e], tokens ascending.
// One CTA per (8 experts x 256 columns): it scans the 8-expert slice of dl for all
// tokens in chunks of 64 (staged in shared memory) and touches x only for the tokens
// with a nonzero gradient there (about k/E of them per expert for renormalised or
// sigmoid routing); each thread owns one column and 8 accumulators.
constexpr int DW_E = 8, DW_T = 64;
template <typename T>
__global__ void __launch_bounds__(TB)
router_dw_kernel(const float* __restrict__ dl, const T* __restrict__ x, float* __restrict__ dwr,
                 float* __restrict__ db, int N, int E, int d) {
  __shared__ float sl[DW_T][DW_E];
  __shared__ int list[DW_T];
  __shared__ int nlist;
  const int e0 = blockIdx.y * DW_E;
  const int c = blockIdx.x * TB + threadIdx.x;
  float acc[DW_E] = {}, bsum[DW_E] = {};
  for (int t0 = 0; t0 < N; t0 += DW_T) {
    for (int i = threadIdx.x; i < DW_T * DW_E; i += TB) {
      const int r = i / DW_E, e = i % DW_E;
      const int t = t0 + r;
      sl[r][e] = (t < N && e0 + e < E) ? dl[(int64_t)t * E + e0 + e] : 0.0f;
    }
    __syncthreads();
    if (threadIdx.x < 32) {  // tokens of this chunk with any nonzero gradient, ascending
      int n = 0;
      for (int r0 = 0; r0 < DW_T; r0 += 32) {
        const int r = r0 + threadIdx.x;
        bool any = false;
#pragma unroll
        for (int e = 0; e < DW_E; ++e) any |= sl[r][e] != 0.0f;
        const unsigned m = __ballot_sync(0xffffffffu, any);
        if (any) list[n + __popc(m & ((1u << threadIdx.x) - 1u))] = r;
        n += __popc(m);
      }
      if (threadIdx.x == 0) nlist = n;
    }
    __syncthreads();
    const int n = nlist;
    for (int i = 0; i < n; ++i) {
      const int r = list[i];
      const float xv = c < d ? to_f32(x[(int64_t)(t0 + r) * d + c]) : 0.0f;
#pragma unroll
      for (int e = 0; e < DW_E; ++e) {
        acc[e] = fmaf(sl[r][e], xv, acc[e]);
        bsum[e] += sl[r][e];
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int e = 0; e < DW_E; ++e) {
    if (e0 + e >= E) break;
    if (c < d) dwr[(int64_t)(e0 + e) * d + c] = acc[e];
    if (blockIdx.x == 0 && threadIdx.x == 0) db[e0 + e] = bsum[e];
  }
}

template <typename T>
__global__ void __launch_bounds__(TB)
dispatch_bwd_kernel(const T* __restrict__ dxperm, const int32_t* __restrict__ slot_of,
                    const T* __restrict__ dout, const T* __restrict__ dxs,
                    const float* __restrict__ dxr, T* __restrict__ dx, int N, int k, int d) {
  const int units = d / 8;
  for (int t = blockIdx.x; t < N; t += gridDim.x) {
    int slots[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) slots[j] = (j < k) ? slot_of[(int64_t)t * k + j] : -1;
    for (int u = threadIdx.x; u < units; u += TB) {
      float acc[8], tmp[8];
      V8<T>::load(dout + (int64_t)t * d, u, acc);
      if (dxs) {
        V8<T>::load(dxs + (int64_t)t * d, u, tmp);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += tmp[i];
      }
      if (dxr) {
        V8<float>::load(dxr + (int64_t)t * d, u, tmp);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += tmp[i];
      }
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {
        if (slots[j] < 0) continue;
        V8<T>::load(dxperm + (int64_t)slots[j] * d, u, tmp);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += tmp[i];
      }
      V8<T>::store(dx + (int64_t)t * d, u, acc);
    }
  }
}

// Zero the `per` 16-byte vectors of buf[e] for every expert e with no kept rows:
// blockIdx.y = expert; CTAs of experts that have rows return at once.
int grid_rows(int64_t rows) {
  const int64_t g = (int64_t)num_sms() * 4;
  return (int)(rows < g ? (rows > 0 ? rows : 1) : g);
}

}  // namespace

cudaError_t launch_combine_backward(const Cfg& c, const void* dout, const void* yperm,
                                    const int32_t* slot_of, const float* topk_w, void* dyperm,
                                    float* dtopk_w, cudaStream_t s) {
  const int g = grid_rows(c.N);
  if (c.act == MOE_DTYPE_F32)
    combine_bwd_kernel<float><<<g, TB, 0, s>>>(
        static_cast<const float*>(dout), static_cast<const float*>(yperm), slot_of, topk_w,
        static_cast<float*>(dyperm), dtopk_w, c.N, c.k, c.d);
  else
    combine_bwd_kernel<__nv_bfloat16><<<g, TB, 0, s>>>(
        static_cast<const __nv_bfloat16*>(dout), static_cast<const __nv_bfloat16*>(yperm),
        slot_of, topk_w, static_cast<__nv_bfloat16*>(dyperm), dtopk_w, c.N, c.k, c.d);
  return cudaGetLastError();
}

cudaError_t launch_route_backward(const Cfg& c, const void* x, const float* w_router,
                                  const float* logits, const int32_t* topk_idx,
                                  const float* dtopk_w, float* dlogits, float* dx_router,
                                  float* dw_router, float* db_router, void* ws, int* status,
                                  cudaStream_t s) {
  const int wg = (int)((c.N + TB / 32 - 1) / (TB / 32));
  route_bwd_kernel<<<wg < num_sms() * 8 ? wg : num_sms() * 8, TB, 0, s>>>(
      logits, topk_idx, dtopk_w, dlogits, c.N, c.E, c.k, c.score_fn, c.normalize ? 1 : 0);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (dx_router) {
    router_dx_kernel<<<grid_rows(c.N), TB, 0, s>>>(dlogits, w_router, dx_router, c.N, c.E, c.d);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (dw_router && ws && c.act == MOE_DTYPE_BF16 && c.N >= kRouterDwTcTokens)
    return launch_router_dw_tc(c, dlogits, x, dw_router, db_router, ws, status, s);
  if (dw_router) {
    const dim3 grid((c.d + TB - 1) / TB, (c.E + DW_E - 1) / DW_E);
    if (c.act == MOE_DTYPE_F32)
      router_dw_kernel<float><<<grid, TB, 0, s>>>(dlogits, static_cast<const float*>(x),
                                                  dw_router, db_router, c.N, c.E, c.d);
    else
      router_dw_kernel<__nv_bfloat16><<<grid, TB, 0, s>>>(
          dlogits, static_cast<const __nv_bfloat16*>(x), dw_router, db_router, c.N, c.E, c.d);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_dispatch_backward(const Cfg& c, const void* dxperm, const int32_t* slot_of,
                                     const void* dout, const void* dx_shared,
                                     const float* dx_router, void* dx, cudaStream_t s) {
  const int g = grid_rows(c.N);
  if (c.act == MOE_DTYPE_F32)
    dispatch_bwd_kernel<float><<<g, TB, 0, s>>>(
        static_cast<const float*>(dxperm), slot_of, static_cast<const float*>(dout),
        static_cast<const float*>(dx_shared), dx_router, static_cast<float*>(dx), c.N, c.k, c.d);
  else
    dispatch_bwd_kernel<__nv_bfloat16><<<g, TB, 0, s>>>(
        static_cast<const __nv_bfloat16*>(dxperm), slot_of,
        static_cast<const __nv_bfloat16*>(dout), static_cast<const __nv_bfloat16*>(dx_shared),
        dx_router, static_cast<__nv_bfloat16*>(dx), c.N, c.k, c.d);
  return cudaGetLastError();
}

}  // namespace moe
