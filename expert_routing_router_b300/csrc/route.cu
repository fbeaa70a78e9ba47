// route.cu -- router scoring + top-k selection (one fused kernel).
//
// Ultralytics glossary "Expert Parallelism", section "How tokens move between GPUs",
// step 1: the router (a linear layer hidden -> num_experts) scores every token
// against every expert and keeps the k best; step 4: the outputs are later weighted
// by the router scores.  Section "Load balancing and capacity": DeepSeek-V3 adds a
// per-expert bias to the scores that only changes which experts are selected, and
// lets a token reach experts on at most 4 of 8 nodes (group-limited routing).
//
// One CTA owns 32 tokens and all E <= 256 experts, so the whole logits row of a
// token is on chip when its selection runs:
//   phase 1  logits tile [32, E] = x[32, d] . W[E, d]^T in fp32 FMAs (SIMT), d in
//            chunks of 32 staged through shared memory;
//   phase 2  + router bias, logits written out, then one warp per token: score,
//            optional group limit, k rounds of warp-shuffle arg-max, weights.
// Ordering everywhere: larger key first, lower expert (group) index on ties.
#include <float.h>
#include <math.h>

#include "moe_internal.cuh"
#include "sigmoid_fixed.cuh"

namespace moe {
namespace {

constexpr int TM = 32;        // tokens per CTA
constexpr int KC = 32;        // d-chunk
constexpr int THREADS = 256;  // 8 warps
constexpr int MAXJ = kMaxExperts / 32;

struct Best {
  float key;
  int idx;
  float val;
};

// a ranks before b: larger key, or equal key and lower index.
__device__ __forceinline__ bool before(float ka, int ia, float kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

__device__ __forceinline__ Best warp_best(Best b) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float k2 = __shfl_xor_sync(0xffffffffu, b.key, off);
    const int i2 = __shfl_xor_sync(0xffffffffu, b.idx, off);
    const float v2 = __shfl_xor_sync(0xffffffffu, b.val, off);
    if (before(k2, i2, b.key, b.idx)) {
      b.key = k2;
      b.idx = i2;
      b.val = v2;
    }
  }
  return b;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

struct RouteParams {
  int N, d, E, k, score_fn, normalize, G, TG;
};

// Selection for the tokens of one tile whose logits sit in shared memory
// (lt[r * EP + e] for r < rows_tile), one warp per token: score, optional group limit, k
// rounds of warp-shuffle arg-max, combine weights.  All threads of the CTA call it.
__device__ void select_tile(float* lt, int EP, int t0, int rows_tile, const RouteParams& p,
                            const float* __restrict__ sel_bias, int32_t* __restrict__ topk_idx,
                            float* __restrict__ topk_w) {
  const int E = p.E;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int EJ = (E + 31) / 32;
  const int gs = E / p.G;
  for (int r = warp; r < rows_tile; r += THREADS / 32) {
    const int t = t0 + r;
    if (t >= p.N) break;
    float* row = lt + r * EP;
    float key[MAXJ], val[MAXJ];
    uint32_t valid = 0;
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) {
      const int e = lane + 32 * j;
      key[j] = -INFINITY;
      val[j] = 0.0f;
      if (j < EJ && e < E) {
        const float l = row[e];
        if (p.score_fn == MOE_SCORE_SIGMOID) {
          const float s = sigmoid_fixed(l);
          val[j] = s;
          key[j] = sel_bias ? __fadd_rn(s, sel_bias[e]) : s;
        } else {
          val[j] = l;
          key[j] = l;
        }
        valid |= 1u << j;
      }
    }
    if (p.G > 1) {
      // ranking keys into the row (the warp owns it), then lane g < G scans group g
      __syncwarp();
#pragma unroll
      for (int j = 0; j < MAXJ; ++j) {
        const int e = lane + 32 * j;
        if (j < EJ && e < E) row[e] = key[j];
      }
      __syncwarp();
      float gscore = -INFINITY;
      int gid = INT_MAX;
      if (lane < p.G) {
        float a = -INFINITY, c = -INFINITY;  // largest, second largest
        for (int i = 0; i < gs; ++i) {
          const float v = row[lane * gs + i];
          if (v > a) {
            c = a;
            a = v;
          } else if (v > c) {
            c = v;
          }
        }
        gscore = (gs >= 2) ? __fadd_rn(a, c) : a;
        gid = lane;
      }
      uint32_t gmask = 0;
      for (int it = 0; it < p.TG; ++it) {
        Best bb = warp_best(Best{gscore, gid, 0.0f});
        gmask |= 1u << bb.idx;
        if (gid == bb.idx) {
          gscore = -INFINITY;
          gid = INT_MAX;
        }
      }
#pragma unroll
      for (int j = 0; j < MAXJ; ++j) {
        const int e = lane + 32 * j;
        if ((valid >> j & 1u) && !((gmask >> (e / gs)) & 1u)) valid &= ~(1u << j);
      }
    }
    // k rounds of arg-max
    int sel_idx = -1;
    float sel_val = 0.0f;
    for (int it = 0; it < p.k; ++it) {
      Best mine{-INFINITY, INT_MAX, 0.0f};
#pragma unroll
      for (int j = 0; j < MAXJ; ++j) {
        if ((valid >> j) & 1u) {
          const int e = lane + 32 * j;
          if (before(key[j], e, mine.key, mine.idx)) mine = Best{key[j], e, val[j]};
        }
      }
      const Best bb = warp_best(mine);
      if (bb.idx < E && (bb.idx & 31) == lane) valid &= ~(1u << (bb.idx >> 5));
      if (lane == it) {
        sel_idx = bb.idx;
        sel_val = bb.val;
      }
    }
    // weights
    float w;
    if (p.score_fn == MOE_SCORE_SIGMOID) {
      const float ssum = warp_sum(lane < p.k ? sel_val : 0.0f);
      w = p.normalize ? sel_val / ssum : sel_val;
    } else {
      float m = -INFINITY;
#pragma unroll
      for (int j = 0; j < MAXJ; ++j)
        if (j < EJ && lane + 32 * j < E) m = fmaxf(m, val[j]);
      m = warp_max(m);
      float z = 0.0f;
#pragma unroll
      for (int j = 0; j < MAXJ; ++j)
        if (j < EJ && lane + 32 * j < E) z += expf(val[j] - m);
      z = warp_sum(z);
      const float pe = (lane < p.k) ? expf(sel_val - m) : 0.0f;
      const float zsel = warp_sum(pe);
      w = p.normalize ? pe / zsel : pe / z;
    }
    if (lane < p.k) {
      topk_idx[(int64_t)t * p.k + lane] = sel_idx;
      topk_w[(int64_t)t * p.k + lane] = w;
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(THREADS)
route_kernel(const T* __restrict__ x, const float* __restrict__ W, const float* __restrict__ b,
             const float* __restrict__ sel_bias, float* __restrict__ logits,
             int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, RouteParams p) {
  extern __shared__ float smem[];
  const int E = p.E;
  const int EP = E + 1;                       // padded row of the logits tile
  float* xs = smem;                           // [TM][KC + 1]
  float* ws = smem + TM * (KC + 1);           // [E][KC + 1]
  float* lt = smem;                           // phase 2: [TM][E + 1] (reuses phase-1 space)

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int t0 = blockIdx.x * TM;
  const int EJ = (E + 31) / 32;

  // ---------------- phase 1: logits tile
  float acc[4][MAXJ];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) acc[i][j] = 0.0f;

  for (int k0 = 0; k0 < p.d; k0 += KC) {
    __syncthreads();
    for (int q = tid; q < TM * KC; q += THREADS) {
      const int r = q / KC, c = q % KC;
      const int t = t0 + r, kk = k0 + c;
      xs[r * (KC + 1) + c] = (t < p.N && kk < p.d) ? to_f32(x[(int64_t)t * p.d + kk]) : 0.0f;
    }
    for (int q = tid; q < E * KC; q += THREADS) {
      const int e = q / KC, c = q % KC;
      const int kk = k0 + c;
      ws[e * (KC + 1) + c] = (kk < p.d) ? W[(int64_t)e * p.d + kk] : 0.0f;
    }
    __syncthreads();
#pragma unroll 8
    for (int c = 0; c < KC; ++c) {
      float xv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) xv[i] = xs[(warp * 4 + i) * (KC + 1) + c];
#pragma unroll
      for (int j = 0; j < MAXJ; ++j) {
        if (j < EJ) {
          const int e = lane + 32 * j;
          const float wv = (e < E) ? ws[e * (KC + 1) + c] : 0.0f;
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[i][j] = fmaf(xv[i], wv, acc[i][j]);
        }
      }
    }
  }
  __syncthreads();

  // ---------------- phase 2a: bias, logits out
#pragma unroll
  for (int j = 0; j < MAXJ; ++j) {
    const int e = lane + 32 * j;
    if (j < EJ && e < E) {
      const float be = b ? b[e] : 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) lt[(warp * 4 + i) * EP + e] = acc[i][j] + be;
    }
  }
  __syncthreads();
  for (int q = tid; q < TM * E; q += THREADS) {
    const int r = q / E, e = q % E;
    const int t = t0 + r;
    if (t < p.N) logits[(int64_t)t * E + e] = lt[r * EP + e];
  }
  __syncthreads();  // rows are overwritten with ranking keys below

  select_tile(lt, EP, t0, TM, p, sel_bias, topk_idx, topk_w);
}

// Router logits from the tensor-core path: fixed-order sum of the K slices plus the
// router bias, written out, then the same selection as the SIMT path.  TS tokens per
// CTA: 32, or 8 for small batches, whose few token tiles the GEMM splits into many K
// slices (more CTAs share the slice sums).
template <int TS>
__global__ void __launch_bounds__(THREADS, 4)
select_kernel(const float* __restrict__ partial, int nsplit, int Epad, const float* __restrict__ b,
              const float* __restrict__ sel_bias, float* __restrict__ logits,
              int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, RouteParams p) {
  pdl_wait();  // decode-sized batches: a dependent of the logits kernel, which has completed
  extern __shared__ float smem[];
  const int E = p.E, EP = E + 1;
  float* lt = smem;
  const int t0 = blockIdx.x * TS;
  const int rows = min(TS, p.N - t0);
  if (nsplit == 1) {
    // one slice: each thread moves whole elements (bias added, written out)
    for (int q = threadIdx.x; q < rows * E; q += THREADS) {
      const int r = q / E, e = q - r * E;
      const float o = __ldg(partial + (int64_t)(t0 + r) * Epad + e) + (b ? b[e] : 0.0f);
      lt[r * EP + e] = o;
      logits[(int64_t)(t0 + r) * E + e] = o;
    }
  } else {
    // Thread c (< E <= THREADS) owns column c of the tile and adds the K slices into
    // it slice by slice: its TS loads of one slice are independent, so a slice costs
    // about one memory latency; the additions run in slice order 0, 1, ..., nsplit-1.
    static_assert(kMaxExperts <= THREADS, "one thread per expert column");
    const int col = threadIdx.x;
    if (col < E) {
      const float bc = b ? b[col] : 0.0f;
      for (int sp = 0; sp < nsplit; ++sp) {
        const float* ps = partial + ((int64_t)sp * p.N + t0) * Epad + col;
        float v[TS];
#pragma unroll
        for (int r = 0; r < TS; ++r) v[r] = r < rows ? __ldg(ps + (int64_t)r * Epad) : 0.0f;
#pragma unroll
        for (int r = 0; r < TS; ++r)
          if (r < rows) lt[r * EP + col] = sp == 0 ? v[r] : lt[r * EP + col] + v[r];
      }
#pragma unroll
      for (int r = 0; r < TS; ++r) {
        if (r < rows) {
          const float o = lt[r * EP + col] + bc;
          lt[r * EP + col] = o;
          logits[(int64_t)(t0 + r) * E + col] = o;
        }
      }
    }
  }
  __syncthreads();
  select_tile(lt, EP, t0, rows, p, sel_bias, topk_idx, topk_w);
}

}  // namespace

// Few tokens (decode): logits straight from the fp32 weight on the CUDA cores.  One
// CTA per expert keeps its slice of that expert's weight row in registers and runs it
// against every token (at most kSmallRouteTokens), fp32 FMAs, then a fixed-order block
// sum; the partial-logit layout is the tensor-core path's with one slice, so the same
// select_kernel adds the bias and selects.  The weight is read once and nothing is
// re-split per call (the tensor-core path rewrites the 3-term bf16 split every call).
constexpr int kSmallRouteTokens = 16;
// Batches up to this many tokens select with 8-token tiles (see select_kernel).
constexpr int kSmallSelectTokens = 4096;

__global__ void __launch_bounds__(THREADS)
route_small_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ W,
                   float* __restrict__ partial, int N, int d, int Epad) {
  pdl_trigger();  // the selection kernel may be scheduled now; it waits for this one
  __shared__ float red[THREADS / 32][kSmallRouteTokens];
  const int e = blockIdx.x;
  const int units = d / 8;
  float acc[kSmallRouteTokens];
#pragma unroll
  for (int t = 0; t < kSmallRouteTokens; ++t) acc[t] = 0.0f;
  for (int u = threadIdx.x; u < units; u += THREADS) {
    const float4* wp = reinterpret_cast<const float4*>(W + (int64_t)e * d) + 2 * u;
    const float4 w0 = wp[0], w1 = wp[1];
    const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int t = 0; t < kSmallRouteTokens; ++t) {
      if (t >= N) break;
      const uint4 v = reinterpret_cast<const uint4*>(x + (int64_t)t * d)[u];
      const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[t] = fmaf(w[2 * i], __uint_as_float(q[i] << 16), acc[t]);
        acc[t] = fmaf(w[2 * i + 1], __uint_as_float(q[i] & 0xffff0000u), acc[t]);
      }
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int t = 0; t < kSmallRouteTokens; ++t) {
    float v = acc[t];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) red[warp][t] = v;
  }
  __syncthreads();
  if (threadIdx.x < N) {
    float v = 0.0f;
    for (int w8 = 0; w8 < THREADS / 32; ++w8) v += red[w8][threadIdx.x];
    partial[(int64_t)threadIdx.x * Epad + e] = v;
  }
}

cudaError_t launch_route(const Cfg& c, const void* x, const float* w_router, const float* b_router,
                         const float* sel_bias, float* logits, int32_t* topk_idx, float* topk_w,
                         void* ws_split, float* partial, int* status, cudaStream_t s) {
  RouteParams p{c.N, c.d, c.E, c.k, c.score_fn, c.normalize, c.G, c.TG};
  const dim3 grid((c.N + TM - 1) / TM);
  const size_t sm_sel = (size_t)TM * (c.E + 1) * sizeof(float);
  if (c.act == MOE_DTYPE_F32) {
    // fp32 hidden states: fp32 FMAs on the CUDA cores, selection fused
    const size_t sm1 = (size_t)(TM * (KC + 1) + c.E * (KC + 1)) * sizeof(float);
    const size_t smem = sm1 > sm_sel ? sm1 : sm_sel;
    auto kern = route_kernel<float>;
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    kern<<<grid, THREADS, smem, s>>>(static_cast<const float*>(x), w_router, b_router, sel_bias,
                                     logits, topk_idx, topk_w, p);
    return cudaGetLastError();
  }
  const RouterPlan rp = router_plan(c);
  int nsplit = rp.nsplit;
  if (c.N <= kSmallRouteTokens) {
    // decode-sized batches: fp32 dot products on the CUDA cores, one slice
    route_small_kernel<<<c.E, THREADS, 0, s>>>(static_cast<const __nv_bfloat16*>(x), w_router,
                                                partial, c.N, c.d, rp.Epad);
    nsplit = 1;
  } else {
    // bf16 hidden states: tensor-core GEMM over the 3-term bf16 split of the weight
    cudaError_t e = launch_router_gemm(c, rp, x, w_router, ws_split, partial, status, s);
    if (e != cudaSuccess) return e;
  }
  if (c.N <= kSmallSelectTokens) {
    constexpr int TS = 8;
    const size_t sm = (size_t)TS * (c.E + 1) * sizeof(float);
    if (c.N <= kSmallRouteTokens) {
      // a programmatic dependent of the CUDA-core logits kernel
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      return launch_dependent(select_kernel<TS>, dim3((c.N + TS - 1) / TS), dim3(THREADS), sm,
                              s, static_cast<const float*>(partial), nsplit, rp.Epad, b_router,
                              sel_bias, logits, topk_idx, topk_w, p);
    }
    select_kernel<TS><<<(c.N + TS - 1) / TS, THREADS, sm, s>>>(
        partial, nsplit, rp.Epad, b_router, sel_bias, logits, topk_idx, topk_w, p);
    return cudaGetLastError();
  }
  if (sm_sel > 48 * 1024)
    cudaFuncSetAttribute(select_kernel<TM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sm_sel);
  select_kernel<TM><<<grid, THREADS, sm_sel, s>>>(partial, nsplit, rp.Epad, b_router, sel_bias,
                                                  logits, topk_idx, topk_w, p);
  return cudaGetLastError();
}

}  // namespace moe
