// payload_q8.cu -- INT8 all-to-all payload: quantise on send, dequantise on receive.
//
// bowenzhou.top note "专家并行", section "深入推导：all-to-all 通信模型与 DeepSeek-V3 的
// EP 配置" (DeepSeek-V3's two-level EP): INT8-quantised communication halves the
// all-to-all traffic again.  Format (the pages fix none; symmetric, one fp32 scale
// per row):
//   s   = max_i |v_i| / 127                 (fp32 divide, round to nearest)
//   r   = 1 / s                              (fp32 divide, once per row)
//   q_i = rint(v_i * r) clamped to +-127     (fp32 multiply, round half to even)
//   all-zero row: s = 0, q = 0
//   received value = (float)q_i * s          (one fp32 multiply), rounded once to the
//                                            activation type
// A row of d activations travels as d bytes + one 4-byte scale instead of 2d (bf16)
// or 4d (fp32) bytes.
//
// Kernels (all HBM-bound, one CTA per row, grid-stride over rows):
//   permute_q8_kernel   dispatch side: reads each kept token's row once, finds its
//                       absolute maximum (block reduction), writes the codes and the
//                       scale to every kept slot of that token
//   quant_rows_kernel   expert side of the return trip: the same quantisation of the
//                       send-buffer rows that hold an assignment (perm_src >= 0)
//   dequant_rows_kernel receiver side: codes * scale back to the activation type
//   combine_q8_kernel   combine reading the INT8 return payload: acc = residual
//                       (+ shared) + sum_j w_j * (q * s_j), fp32, j ascending
// The quantising kernels keep a thread's units of a row in registers between the
// max pass and the code pass and overlap one row's stores with the next row's loads;
// rows longer than the register cache are read a second time (from L1/L2).  Grids
// are one wave of resident CTAs (occupancy query), each walking its rows.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int TQ = 256;          // threads per CTA of the kernels without a row reduction
constexpr int TR = 128;          // threads per CTA of the quantising kernels (one row each;
                                 // small CTAs keep more rows in flight per SM)
constexpr int kCacheUnits = 8;   // register-cached units per thread (8192 bf16 per row)

__device__ __forceinline__ uint2 ld_stream_u2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}

// 8 consecutive activations <-> 8 floats.  Unit u of a row starts at element 8u.
template <typename T>
struct Unit;
template <>
struct Unit<__nv_bfloat16> {
  using Raw = uint4;
  __device__ static Raw load_raw(const void* row, int u, bool stream) {
    const uint4* p = static_cast<const uint4*>(row) + u;
    return stream ? ld_stream_u4(p) : *p;
  }
  __device__ static void widen(const Raw& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static void load(const void* row, int u, float* f, bool stream) {
    widen(load_raw(row, u, stream), f);
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
struct Unit<float> {
  struct Raw {
    uint4 a, b;
  };
  __device__ static Raw load_raw(const void* row, int u, bool stream) {
    const uint4* p = static_cast<const uint4*>(row) + 2 * u;
    Raw r;
    r.a = stream ? ld_stream_u4(p) : p[0];
    r.b = stream ? ld_stream_u4(p + 1) : p[1];
    return r;
  }
  __device__ static void widen(const Raw& r, float* f) {
    f[0] = __uint_as_float(r.a.x);
    f[1] = __uint_as_float(r.a.y);
    f[2] = __uint_as_float(r.a.z);
    f[3] = __uint_as_float(r.a.w);
    f[4] = __uint_as_float(r.b.x);
    f[5] = __uint_as_float(r.b.y);
    f[6] = __uint_as_float(r.b.z);
    f[7] = __uint_as_float(r.b.w);
  }
  __device__ static void load(const void* row, int u, float* f, bool stream) {
    widen(load_raw(row, u, stream), f);
  }
  __device__ static void store(void* row, int u, const float* f) {
    uint4* p = static_cast<uint4*>(row) + 2 * u;
    p[0] = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
    p[1] = make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]),
                      __float_as_uint(f[7]));
  }
};

// Code of v for a row with reciprocal scale inv = 1/s (inv = 0 for an all-zero row:
// every code is 0).  One fp32 multiply, round half to even, clamp.
__device__ __forceinline__ uint32_t code_byte(float v, float inv) {
  int c = __float2int_rn(__fmul_rn(v, inv));
  c = max(-127, min(127, c));
  return static_cast<uint32_t>(c) & 0xffu;
}

// Reciprocal of a row's scale, once per row (fp32 divide, round to nearest).
__device__ __forceinline__ float scale_inverse(float s) {
  return s > 0.0f ? __fdiv_rn(1.0f, s) : 0.0f;
}

// 8 codes, byte i = element i.
__device__ __forceinline__ uint2 pack_codes(const float* f, float inv) {
  uint2 r;
  r.x = code_byte(f[0], inv) | (code_byte(f[1], inv) << 8) | (code_byte(f[2], inv) << 16) |
        (code_byte(f[3], inv) << 24);
  r.y = code_byte(f[4], inv) | (code_byte(f[5], inv) << 8) | (code_byte(f[6], inv) << 16) |
        (code_byte(f[7], inv) << 24);
  return r;
}

__device__ __forceinline__ void unpack_codes(uint2 v, float* f) {
  const uint32_t w[2] = {v.x, v.y};
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int i = 0; i < 4; ++i)
      f[4 * h + i] = static_cast<float>(static_cast<int8_t>((w[h] >> (8 * i)) & 0xffu));
}

// Maximum over the CTA (all threads call it; red holds 33 floats).
__device__ float block_max(float m, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[32] = m;
  }
  __syncthreads();
  m = red[32];
  __syncthreads();  // red is reused by the next row
  return m;
}

// Quantise one row held at `row` (act type T, `units` units): returns the scale and
// calls emit(u, packed codes) for every unit.  First pass: absolute maximum (the
// first kCacheUnits units of each thread stay in registers); second pass: codes.
template <typename T, typename Emit>
__device__ float quantise_row(const void* row, int units, float* red, Emit emit) {
  typename Unit<T>::Raw cache[kCacheUnits];
  float m = 0.0f;
#pragma unroll
  for (int r = 0; r < kCacheUnits; ++r) {
    const int u = threadIdx.x + r * TR;
    if (u < units) {
      float f[8];
      cache[r] = Unit<T>::load_raw(row, u, false);
      Unit<T>::widen(cache[r], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
    }
  }
  for (int u = threadIdx.x + kCacheUnits * TR; u < units; u += TR) {
    float f[8];
    Unit<T>::load(row, u, f, false);
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
  }
  const float amax = block_max(m, red);
  const float s = __fdiv_rn(amax, 127.0f);
  const float inv = scale_inverse(s);
#pragma unroll
  for (int r = 0; r < kCacheUnits; ++r) {
    const int u = threadIdx.x + r * TR;
    if (u < units) {
      float f[8];
      Unit<T>::widen(cache[r], f);
      emit(u, pack_codes(f, inv));
    }
  }
  for (int u = threadIdx.x + kCacheUnits * TR; u < units; u += TR) {
    float f[8];
    Unit<T>::load(row, u, f, false);
    emit(u, pack_codes(f, inv));
  }
  return s;
}

// Register-cached units per thread for the pipelined path: 8 bf16 units (8192 bf16
// per row at 128 threads) or 4 fp32 units (4096 fp32 per row).
template <typename T>
struct CacheUnits {
  static constexpr int value = sizeof(T) == 2 ? 8 : 4;
};

// The rows one CTA quantises (a grid-stride walk), software-pipelined: once the
// current row's maximum is known, the next row's loads are issued before the current
// row's codes are written, so one row's stores overlap the next row's loads.  Rows
// longer than the register cache take the two-pass quantise_row instead.  Src gives
//   next(r)   first row >= r that is sent (or >= its row count)
//   begin(r)  row r becomes current (per-row state, e.g. its slots)
//   row(r)    pointer to row r
//   store(u, codes), finish(s)   outputs of the current row
template <typename T, typename Src>
__device__ void quantise_rows(Src& src, int64_t rows, int units, float* red) {
  constexpr int CU = CacheUnits<T>::value;
  using Raw = typename Unit<T>::Raw;
  if (units > CU * TR) {
    for (int64_t r = src.next(blockIdx.x); r < rows; r = src.next(r + gridDim.x)) {
      src.begin(r);
      const float sc = quantise_row<T>(src.row(r), units, red,
                                       [&](int u, uint2 codes) { src.store(u, codes); });
      src.finish(sc);
    }
    return;
  }
  Raw cur[CU], nxt[CU];
  int64_t r = src.next(blockIdx.x);
  if (r < rows) {
#pragma unroll
    for (int i = 0; i < CU; ++i) {
      const int u = threadIdx.x + i * TR;
      if (u < units) cur[i] = Unit<T>::load_raw(src.row(r), u, true);
    }
  }
  while (r < rows) {
    const int64_t rn = src.next(r + gridDim.x);
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < CU; ++i) {
      const int u = threadIdx.x + i * TR;
      if (u < units) {
        float f[8];
        Unit<T>::widen(cur[i], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(f[e]));
      }
    }
    const float sc = __fdiv_rn(block_max(m, red), 127.0f);
    const float inv = scale_inverse(sc);
    if (rn < rows) {
#pragma unroll
      for (int i = 0; i < CU; ++i) {
        const int u = threadIdx.x + i * TR;
        if (u < units) nxt[i] = Unit<T>::load_raw(src.row(rn), u, true);
      }
    }
    src.begin(r);
#pragma unroll
    for (int i = 0; i < CU; ++i) {
      const int u = threadIdx.x + i * TR;
      if (u < units) {
        float f[8];
        Unit<T>::widen(cur[i], f);
        src.store(u, pack_codes(f, inv));
      }
    }
    src.finish(sc);
#pragma unroll
    for (int i = 0; i < CU; ++i) cur[i] = nxt[i];
    r = rn;
  }
}

// Dispatch side: token rows, each written to every slot it was kept in.
template <typename T>
struct TokenRows {
  const T* x;
  int8_t* xq;
  float* xscale;
  const int32_t* slot_of;
  int N, k, d;
  int slots[kMaxTopK];
  __device__ int64_t next(int64_t t) const {
    for (; t < N; t += gridDim.x) {  // skip tokens whose every choice was dropped
      for (int j = 0; j < k; ++j)
        if (slot_of[t * k + j] >= 0) return t;
    }
    return N;
  }
  __device__ void begin(int64_t t) {
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) slots[j] = (j < k) ? slot_of[t * k + j] : -1;
  }
  __device__ const T* row(int64_t t) const { return x + t * d; }
  __device__ void store(int u, uint2 codes) {
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (slots[j] >= 0) reinterpret_cast<uint2*>(xq + (int64_t)slots[j] * d)[u] = codes;
  }
  __device__ void finish(float sc) {
    if (threadIdx.x == 0) {
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j)
        if (slots[j] >= 0) xscale[slots[j]] = sc;
    }
  }
};

// Return side: send-buffer rows that hold an assignment, quantised in place of row r.
template <typename T>
struct SendRows {
  const T* in;
  const int32_t* perm_src;
  int8_t* q;
  float* scale;
  int64_t rows;
  int d;
  int64_t cur;
  __device__ int64_t next(int64_t r) const {
    while (r < rows && perm_src[r] < 0) r += gridDim.x;  // padding rows hold nothing
    return r < rows ? r : rows;
  }
  __device__ void begin(int64_t r) { cur = r; }
  __device__ const T* row(int64_t r) const { return in + r * d; }
  __device__ void store(int u, uint2 codes) { reinterpret_cast<uint2*>(q + cur * d)[u] = codes; }
  __device__ void finish(float sc) {
    if (threadIdx.x == 0) scale[cur] = sc;
  }
};

template <typename T>
__global__ void __launch_bounds__(TR)
permute_q8_kernel(const T* __restrict__ x, int8_t* __restrict__ xq, float* __restrict__ xscale,
                  const int32_t* __restrict__ slot_of, int N, int k, int d) {
  __shared__ float red[33];
  TokenRows<T> src{x, xq, xscale, slot_of, N, k, d, {}};
  quantise_rows<T>(src, N, d / 8, red);
}

template <typename T>
__global__ void __launch_bounds__(TR)
quant_rows_kernel(const T* __restrict__ in, const int32_t* __restrict__ perm_src,
                  int8_t* __restrict__ q, float* __restrict__ scale, int64_t rows, int d) {
  __shared__ float red[33];
  SendRows<T> src{in, perm_src, q, scale, rows, d, 0};
  quantise_rows<T>(src, rows, d / 8, red);
}

template <typename T>
__global__ void __launch_bounds__(TQ)
dequant_rows_kernel(const int8_t* __restrict__ q, const float* __restrict__ scale,
                    const int32_t* __restrict__ perm_src, T* __restrict__ out, int64_t rows,
                    int d) {
  const int units = d / 8;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    if (perm_src[r] < 0) continue;
    const float s = scale[r];
    const int8_t* qrow = q + r * d;
    T* orow = out + r * d;
    for (int u = threadIdx.x; u < units; u += TQ) {
      float f[8];
      unpack_codes(ld_stream_u2(qrow + 8 * (int64_t)u), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(f[i], s);
      Unit<T>::store(orow, u, f);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(TQ)
combine_q8_kernel(const int8_t* __restrict__ yq, const float* __restrict__ yscale,
                  const int32_t* __restrict__ slot_of, const float* __restrict__ topk_w,
                  const T* __restrict__ residual, const T* __restrict__ yshared,
                  T* __restrict__ out, int N, int k, int d) {
  const int units = d / 8;
  for (int t = blockIdx.x; t < N; t += gridDim.x) {
    int slots[kMaxTopK];
    float w[kMaxTopK], sc[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      slots[j] = (j < k) ? slot_of[(int64_t)t * k + j] : -1;
      w[j] = (j < k) ? topk_w[(int64_t)t * k + j] : 0.0f;
      sc[j] = slots[j] >= 0 ? yscale[slots[j]] : 0.0f;
    }
    const T* rrow = residual ? residual + (int64_t)t * d : nullptr;
    const T* srow = yshared ? yshared + (int64_t)t * d : nullptr;
    T* orow = out + (int64_t)t * d;
    for (int u = threadIdx.x; u < units; u += TQ) {
      uint2 raw[kMaxTopK];
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j)
        if (slots[j] >= 0) raw[j] = ld_stream_u2(yq + (int64_t)slots[j] * d + 8 * (int64_t)u);
      float acc[8], tmp[8];
      if (rrow) {
        Unit<T>::load(rrow, u, acc, true);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
      }
      if (srow) {
        Unit<T>::load(srow, u, tmp, true);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += tmp[i];
      }
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {
        if (slots[j] >= 0) {
          unpack_codes(raw[j], tmp);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(w[j], __fmul_rn(tmp[i], sc[j]), acc[i]);
        }
      }
      Unit<T>::store(orow, u, acc);
    }
  }
}

// One wave of resident CTAs (every CTA then walks its rows; a second partial wave
// would double the time of the rows it holds), capped by the row count.
// The occupancy query runs once per kernel and device (not inside every launch, so
// a launch under stream capture makes no extra runtime call).
template <auto kernel, int threads = TQ>
int row_grid(int64_t rows) {
  static int cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] == 0) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    cached[dev] = per_sm;
  }
  const int64_t g = (int64_t)num_sms() * cached[dev];
  return (int)(rows < g ? (rows > 0 ? rows : 1) : g);
}

}  // namespace

cudaError_t launch_dispatch_q8(const Cfg& c, const int32_t* topk_idx, const void* x, int8_t* xq,
                               float* xscale, int32_t* expert_counts, int32_t* kept_counts,
                               int32_t* expert_start, int32_t* rank_counts, int32_t* rank_offsets,
                               int32_t* slot_of, int32_t* perm_src, int32_t* num_kept,
                               int32_t* chunk_hist, cudaStream_t s) {
  // counting, capacity and slot assignment exactly as the activation-typed dispatch
  cudaError_t e = launch_dispatch(c, topk_idx, nullptr, nullptr, expert_counts, kept_counts,
                                  expert_start, rank_counts, rank_offsets, slot_of, perm_src,
                                  num_kept, chunk_hist, s);
  if (e != cudaSuccess) return e;
  if (c.act == MOE_DTYPE_F32) {
    const int g = row_grid<permute_q8_kernel<float>, TR>(c.N);
    permute_q8_kernel<float><<<g, TR, 0, s>>>(static_cast<const float*>(x), xq, xscale, slot_of,
                                              c.N, c.k, c.d);
  } else {
    const int g = row_grid<permute_q8_kernel<__nv_bfloat16>, TR>(c.N);
    permute_q8_kernel<__nv_bfloat16><<<g, TR, 0, s>>>(static_cast<const __nv_bfloat16*>(x), xq,
                                                      xscale, slot_of, c.N, c.k, c.d);
  }
  return cudaGetLastError();
}

cudaError_t launch_quant_rows(const Cfg& c, const void* in, const int32_t* perm_src, int8_t* q,
                              float* scale, cudaStream_t s) {
  if (c.act == MOE_DTYPE_F32) {
    const int g = row_grid<quant_rows_kernel<float>, TR>(c.send_rows);
    quant_rows_kernel<float><<<g, TR, 0, s>>>(static_cast<const float*>(in), perm_src, q, scale,
                                              c.send_rows, c.d);
  } else {
    const int g = row_grid<quant_rows_kernel<__nv_bfloat16>, TR>(c.send_rows);
    quant_rows_kernel<__nv_bfloat16><<<g, TR, 0, s>>>(static_cast<const __nv_bfloat16*>(in),
                                                      perm_src, q, scale, c.send_rows, c.d);
  }
  return cudaGetLastError();
}

cudaError_t launch_dequant_rows(const Cfg& c, const int8_t* q, const float* scale,
                                const int32_t* perm_src, void* out, cudaStream_t s) {
  if (c.act == MOE_DTYPE_F32) {
    const int g = row_grid<dequant_rows_kernel<float>>(c.send_rows);
    dequant_rows_kernel<float><<<g, TQ, 0, s>>>(q, scale, perm_src, static_cast<float*>(out),
                                                c.send_rows, c.d);
  } else {
    const int g = row_grid<dequant_rows_kernel<__nv_bfloat16>>(c.send_rows);
    dequant_rows_kernel<__nv_bfloat16><<<g, TQ, 0, s>>>(
        q, scale, perm_src, static_cast<__nv_bfloat16*>(out), c.send_rows, c.d);
  }
  return cudaGetLastError();
}

cudaError_t launch_combine_q8(const Cfg& c, const int8_t* yq, const float* yscale,
                              const int32_t* slot_of, const float* topk_w, const void* residual,
                              const void* yshared, void* out, cudaStream_t s) {
  if (c.act == MOE_DTYPE_F32) {
    const int g = row_grid<combine_q8_kernel<float>>(c.N);
    combine_q8_kernel<float><<<g, TQ, 0, s>>>(yq, yscale, slot_of, topk_w,
                                              static_cast<const float*>(residual),
                                              static_cast<const float*>(yshared),
                                              static_cast<float*>(out), c.N, c.k, c.d);
  } else {
    const int g = row_grid<combine_q8_kernel<__nv_bfloat16>>(c.N);
    combine_q8_kernel<__nv_bfloat16><<<g, TQ, 0, s>>>(
        yq, yscale, slot_of, topk_w, static_cast<const __nv_bfloat16*>(residual),
        static_cast<const __nv_bfloat16*>(yshared), static_cast<__nv_bfloat16*>(out), c.N, c.k,
        c.d);
  }
  return cudaGetLastError();
}

}  // namespace moe
