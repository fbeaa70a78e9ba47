// ffn_simt.cu -- grouped SwiGLU expert FFN on CUDA cores (fp32 activations).
//
// Ultralytics glossary "Expert Parallelism", section "How tokens move between GPUs",
// step 3: every rank runs its local experts on the rows it received.  Each expert is
// a SwiGLU feed-forward block h = silu(X Wg^T) * (X Wu^T), Y = h Wd^T;
// fudan-mlsys-cn chapter 10, section 10.5: a shared expert sees every token.
//
// fp32 products need fp32 FMAs (a TF32 tensor-core pass would miss a 1e-4 relative
// bound), so this path tiles the two grouped GEMMs for the SIMT pipes:
//   G1  h[rows, F]  = silu(X . Wg^T) * (X . Wu^T)    64x64 tile, gate+up together
//   G2  Y[rows, d]  = h . Wd^T                       64x64 tile
// Segments: routed expert e owns xperm rows [expert_start[e], +kept_counts[e]);
// the shared expert (if any) is segment E over the N rows of x.  The grid covers
// the worst-case tile count; each CTA resolves its (segment, row tile) from the
// device-side counts, so nothing is read back to the host.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, TS = 256;

struct Seg {
  int seg, m0, rows, a_row;  // segment id, first row in segment, valid rows, A row base
};

// Resolve blockIdx.y into (segment, row tile).  Returns false past the last tile.
__device__ bool resolve_tile(const int32_t* expert_start, const int32_t* kept_counts, int E,
                             int n_shared, int* sm_prefix, Seg* out) {
  const int nseg = E + (n_shared > 0 ? 1 : 0);
  if (threadIdx.x < 32) {
    int base = 0;
    for (int s0 = 0; s0 < nseg; s0 += 32) {
      const int s = s0 + threadIdx.x;
      int v = 0;
      if (s < nseg) {
        const int cnt = (s < E) ? kept_counts[s] : n_shared;
        v = (cnt + BM - 1) / BM;
      }
      int incl = v;
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if ((int)threadIdx.x >= off) incl += y;
      }
      if (s < nseg) sm_prefix[s] = base + incl - v;
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (threadIdx.x == 0) sm_prefix[nseg] = base;
  }
  __syncthreads();
  const int tile = blockIdx.y;
  if (tile >= sm_prefix[nseg]) return false;
  int lo = 0, hi = nseg - 1;  // last s with prefix[s] <= tile
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sm_prefix[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  const int s = lo;
  const int cnt = (s < E) ? kept_counts[s] : n_shared;
  out->seg = s;
  out->m0 = (tile - sm_prefix[s]) * BM;
  out->rows = min(BM, cnt - out->m0);
  out->a_row = (s < E) ? expert_start[s] : 0;
  return true;
}

template <typename T>
__device__ __forceinline__ void load4(const T* p, float* f);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float* f) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float* f) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xffff0000u);
  f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xffff0000u);
}

// Stage a [64 x 16] slice of row-major M (rows r0.., cols k0..) transposed into
// S[16][64+4]; rows >= nrows or cols >= K read as zero.  Requires K % 4 == 0.
template <typename T>
__device__ __forceinline__ void stage(float (*S)[BM + 4], const T* M, int64_t ld, int r0,
                                      int nrows, int k0, int K) {
  const int r = threadIdx.x >> 2, c = (threadIdx.x & 3) * 4;
  float f[4] = {0.f, 0.f, 0.f, 0.f};
  if (r < nrows && k0 + c < K) load4<T>(M + (int64_t)(r0 + r) * ld + k0 + c, f);
#pragma unroll
  for (int i = 0; i < 4; ++i) S[c + i][r] = f[i];
}

template <typename T>
__global__ void __launch_bounds__(TS)
ffn_gate_up_kernel(const T* __restrict__ xperm, const T* __restrict__ x,
                   const int32_t* __restrict__ expert_start, const int32_t* __restrict__ kept_counts,
                   const T* __restrict__ wgu, const T* __restrict__ sgu, T* __restrict__ h,
                   int64_t h_shared_off, int E, int N_shared, int d, int F, int Fs) {
  __shared__ int prefix[kMaxExperts + 2];
  __shared__ float As[BK][BM + 4], Gs[BK][BN + 4], Us[BK][BN + 4];
  Seg sg;
  if (!resolve_tile(expert_start, kept_counts, E, N_shared, prefix, &sg)) return;
  const bool shared = sg.seg == E;
  const int Fx = shared ? Fs : F;
  const int f0 = blockIdx.x * BN;
  if (f0 >= Fx) return;
  const T* A = shared ? x : xperm;
  const T* Wg = shared ? sgu : wgu + (int64_t)sg.seg * 2 * F * d;
  const T* Wu = Wg + (int64_t)Fx * d;
  const int arow = sg.a_row + sg.m0;
  const int nf = min(BN, Fx - f0);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float ag[4][4] = {}, au[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += BK) {
    __syncthreads();
    stage<T>(As, A, d, arow, sg.rows, k0, d);
    stage<T>(Gs, Wg, d, f0, nf, k0, d);
    stage<T>(Us, Wu, d, f0, nf, k0, d);
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], g[4], u[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        g[i] = Gs[kk][tx * 4 + i];
        u[i] = Us[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          ag[i][j] = fmaf(a[i], g[j], ag[i][j]);
          au[i][j] = fmaf(a[i], u[j], au[i][j]);
        }
    }
  }
  T* hb = shared ? h + h_shared_off : h;
  const int hrow0 = shared ? sg.m0 : sg.a_row + sg.m0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty * 4 + i;
    if (r >= sg.rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int f = f0 + tx * 4 + j;
      if (f >= Fx) continue;
      const float g = ag[i][j];
      const float v = g / (1.0f + expf(-g)) * au[i][j];
      hb[(int64_t)(hrow0 + r) * Fx + f] = from_f32<T>(v);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(TS)
ffn_down_kernel(const T* __restrict__ h, const int32_t* __restrict__ expert_start,
                const int32_t* __restrict__ kept_counts, const T* __restrict__ wd,
                const T* __restrict__ sd, T* __restrict__ yperm, T* __restrict__ yshared,
                int64_t h_shared_off, int E, int N_shared, int d, int F, int Fs) {
  __shared__ int prefix[kMaxExperts + 2];
  __shared__ float As[BK][BM + 4], Bs[BK][BN + 4];
  Seg sg;
  if (!resolve_tile(expert_start, kept_counts, E, N_shared, prefix, &sg)) return;
  const bool shared = sg.seg == E;
  const int Fx = shared ? Fs : F;
  const int o0 = blockIdx.x * BN;
  if (o0 >= d) return;
  const T* A = shared ? h + h_shared_off : h;
  const int arow = shared ? sg.m0 : sg.a_row + sg.m0;
  const T* Wd = shared ? sd : wd + (int64_t)sg.seg * d * F;
  const int no = min(BN, d - o0);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < Fx; k0 += BK) {
    __syncthreads();
    stage<T>(As, A, Fx, arow, sg.rows, k0, Fx);
    stage<T>(Bs, Wd, Fx, o0, no, k0, Fx);
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
  }
  T* Y = shared ? yshared : yperm;
  const int yrow0 = shared ? sg.m0 : sg.a_row + sg.m0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty * 4 + i;
    if (r >= sg.rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int o = o0 + tx * 4 + j;
      if (o < d) Y[(int64_t)(yrow0 + r) * d + o] = from_f32<T>(acc[i][j]);
    }
  }
}

template <typename T>
cudaError_t run(const Cfg& c, const void* xperm, const int32_t* expert_start,
                const int32_t* kept_counts, const void* w_gate_up, const void* w_down,
                const void* x, const void* sgu, const void* sd, void* yperm, void* yshared,
                void* h, cudaStream_t s) {
  const int n_shared = c.Fs > 0 ? c.N : 0;
  // worst case: every segment adds at most one partial tile
  const int64_t max_tiles = c.A / BM + c.E + (n_shared + BM - 1) / BM + 1;
  const int64_t h_shared_off = c.send_rows * (int64_t)c.F;
  const int fmax = c.F > c.Fs ? c.F : c.Fs;
  dim3 g1((fmax + BN - 1) / BN, (unsigned)max_tiles);
  ffn_gate_up_kernel<T><<<g1, TS, 0, s>>>(
      static_cast<const T*>(xperm), static_cast<const T*>(x), expert_start, kept_counts,
      static_cast<const T*>(w_gate_up), static_cast<const T*>(sgu), static_cast<T*>(h),
      h_shared_off, c.E, n_shared, c.d, c.F, c.Fs);
  dim3 g2((c.d + BN - 1) / BN, (unsigned)max_tiles);
  ffn_down_kernel<T><<<g2, TS, 0, s>>>(
      static_cast<const T*>(h), expert_start, kept_counts, static_cast<const T*>(w_down),
      static_cast<const T*>(sd), static_cast<T*>(yperm), static_cast<T*>(yshared), h_shared_off,
      c.E, n_shared, c.d, c.F, c.Fs);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ffn_simt(const Cfg& c, const void* xperm, const int32_t* expert_start,
                            const int32_t* kept_counts, const void* w_gate_up, const void* w_down,
                            const void* x, const void* shared_gate_up, const void* shared_down,
                            void* yperm, void* yshared, void* h, cudaStream_t s) {
  if (c.act == MOE_DTYPE_F32)
    return run<float>(c, xperm, expert_start, kept_counts, w_gate_up, w_down, x, shared_gate_up,
                      shared_down, yperm, yshared, h, s);
  return run<__nv_bfloat16>(c, xperm, expert_start, kept_counts, w_gate_up, w_down, x,
                            shared_gate_up, shared_down, yperm, yshared, h, s);
}

}  // namespace moe
