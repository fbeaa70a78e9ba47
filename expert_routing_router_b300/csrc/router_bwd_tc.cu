// router_bwd_tc.cu -- the router's weight gradient on the tensor cores.
//
// Ultralytics glossary "Expert Parallelism", section "How tokens move between GPUs",
// step 1 (a learned router scores every expert: logits = x Wr^T + b), differentiated:
// with dl = dL/dlogits [N, E] fp32 and x [N, d] bf16,
//   dWr [E, d] = dl^T x        db [E] = sum_t dl[t, :]      (fp32 results)
// dWr is a dense contraction over the N tokens.  The fp32 dl is split exactly into
// three bf16 terms (dl = t0 + t1 + t2, each the bf16 rounding of what the previous
// terms leave; 24 mantissa bits in three 8-bit pieces), stacked along K: row t of the
// split array holds [t0 | t1 | t2] of dl[t, :] (each padded to Epad), so
//   dWr[e, c] = sum_{i<3} sum_t t_i[t, e] x[t, c]
// is one GEMM with M = Epad, N = d, K = 3N.  Both operands have their reduction index
// (the token) as the row, so both are loaded MN-major: 64-element x 64-row TMA boxes,
// 128-byte swizzle, descriptors with a leading offset of one box between 64-element
// MN chunks and 1 KiB between 8-row K groups, and both transpose bits set.
// The tensor core's fp32 accumulation truncates, so a long K chain drifts low; the K
// blocks of a tile go round-robin to four TMEM accumulators (each chain a quarter of
// 3N) and the epilogue adds them in a fixed order with round-to-nearest fp32 adds.
// One persistent kernel, one CTA per SM, tiles of 128 experts x 128 columns (the four
// accumulators fill the 512 TMEM columns): warp 0 TMA producer (6-stage ring), warp 1
// TMEM owner and single-thread tcgen05.mma issuer, warps 2-5 epilogue.  Every mbarrier
// wait is bounded (about 2 s) and reports through the status word.
// db is a plain column sum: per 32-expert slice and token slice one partial, then the
// partials in slice order (both passes in a fixed order, so the result is reproducible).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128, BN = 128, BK = 64, STAGES = 6, NACC = 4;
constexpr int BOX_BYTES = 64 * BK * 2;  // 64 MN elements x 64 K rows, 8 KB
constexpr int A_BYTES = BM * BK * 2;    // two boxes
constexpr int B_BYTES = BN * BK * 2;    // two boxes
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr int TMEM_COLS = NACC * BN;    // 512
constexpr uint64_t WAIT_NS = 2000000000ull;
// kind::f16, D fp32, A and B bf16, both MN-major (transpose bits 15 and 16), M 128, N 128
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN) | (1u << 15) | (1u << 16);
constexpr int DB_SLICES = 64;           // token slices of the db column sum

struct DwParams {
  float* dwr;
  int* err;
  int N, E, Epad, d;
};

struct Ctl {
  uint64_t full[STAGES], empty[STAGES], tfull, tempty, drain;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + sizeof(Ctl);

__device__ bool mbar_wait(uint64_t* b, uint32_t parity, Ctl* ctl, int* err, int code) {
  if (mbar_try_wait(b, parity)) return true;
  const uint64_t t0 = now_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(b, parity)) return true;
    if ((i & 63) == 0) {
      if (*(volatile int*)&ctl->abort) return false;
      if (now_ns() - t0 > WAIT_NS) {
        *(volatile int*)&ctl->abort = 1;
        atomicExch(err, code);
        return false;
      }
    }
  }
}

// MN-major 128-byte-swizzle descriptor: start >> 4, leading offset = one 64-element box
// (between MN chunks), stride offset 1 KiB (between 8-row K groups).
__device__ __forceinline__ uint64_t sdesc_mn(uint32_t a) {
  return (uint64_t)((a & 0x3FFFFu) >> 4) | ((uint64_t)(BOX_BYTES >> 4) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// tmA: the split dl [N rows, 3*Epad] bf16; tmB: x [N rows, d] bf16 (64 x 64 boxes).
__global__ void __launch_bounds__(THREADS, 1)
router_dw_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    DwParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + (size_t)STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = p.Epad / BM, nt = (p.d + BN - 1) / BN;
  const int total = mt * nt;
  const int kblk = (p.N + BK - 1) / BK;  // K blocks of one term
  const int nk = 3 * kblk;               // K blocks of a tile (>= 3)
  const int nacc = nk < NACC ? nk : NACC;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    mbar_init(&ctl->tfull, 1);
    mbar_init(&ctl->tempty, 4);
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(&ctl->tmem_base, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      bool ok = true;
      // m tiles fastest: the CTAs of one column tile run together and share x in L2
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const int m0 = (t % mt) * BM, n0 = (t / mt) * BN;
        for (int kb = 0; kb < nk; ++kb) {
          const int term = kb / kblk, r0 = (kb % kblk) * BK;
          if (!mbar_wait(&ctl->empty[stage], phase ^ 1, ctl, p.err, 1)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + (size_t)stage * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          mbar_expect_tx(&ctl->full[stage], STAGE_BYTES);
#pragma unroll
          for (int j = 0; j < 2; ++j)
            tma_load(sa + j * BOX_BYTES, &tmA, &ctl->full[stage], term * p.Epad + m0 + 64 * j, r0);
#pragma unroll
          for (int j = 0; j < 2; ++j)
            tma_load(sb + j * BOX_BYTES, &tmB, &ctl->full[stage], n0 + 64 * j, r0);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {  // let this CTA's copies land before the CTA goes away
        const uint64_t t0 = now_ns();
        for (int s = 0; s < STAGES; ++s)
          if (armed >> s & 1u)
            while (!mbar_try_wait(&ctl->full[s], armed_parity >> s & 1u) &&
                   now_ns() - t0 < WAIT_NS) {
            }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, tphase = 0;
      bool ok = true, issued = false;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        if (!mbar_wait(&ctl->tempty, tphase ^ 1, ctl, p.err, 2)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&ctl->full[stage], phase, ctl, p.err, 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = saddr(smem + (size_t)stage * STAGE_BYTES);
          const uint32_t b0 = a0 + A_BYTES;
          const uint32_t dt = tmem_base + (uint32_t)((kb % NACC) * BN);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma(dt, sdesc_mn(a0 + kk * 2048), sdesc_mn(b0 + kk * 2048), IDESC,
                   (kb >= NACC || kk > 0) ? 1u : 0u);
          issued = true;
          tc_commit(&ctl->empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(&ctl->tfull);
        tphase ^= 1;
      }
      if (issued) {  // every MMA of this thread has finished before TMEM is freed
        tc_commit(&ctl->drain);
        const uint64_t t0 = now_ns();
        while (!mbar_try_wait(&ctl->drain, 0) && now_ns() - t0 < WAIT_NS) {
        }
      }
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2-5)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint32_t tphase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const int m0 = (t % mt) * BM, n0 = (t / mt) * BN;
      if (!mbar_wait(&ctl->tfull, tphase, ctl, p.err, 4)) break;
      tc_fence_after();
      const int e = m0 + q * 32 + lane;  // this thread's expert (TMEM lane)
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16);
      float* orow = p.dwr + (int64_t)e * p.d;
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        uint32_t a[NACC][32];
#pragma unroll
        for (int i = 0; i < NACC; ++i)
          if (i < nacc) tmem_ld32(tb + (uint32_t)(i * BN + c), a[i]);
        tmem_ld_wait(a[0]);
#pragma unroll
        for (int i = 1; i < NACC; ++i) tmem_regs_ready(a[i]);
        if (e < p.E) {
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float s = __uint_as_float(a[0][j]);
#pragma unroll
            for (int i = 1; i < NACC; ++i)
              if (i < nacc) s = __fadd_rn(s, __uint_as_float(a[i][j]));
            v[j] = s;
          }
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const int col = n0 + c + j;
            if (col < p.d)
              *reinterpret_cast<float4*>(orow + col) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->tempty);
      tphase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// The three bf16 terms of every dl value, row t = [t0 | t1 | t2], each Epad wide (zero
// past E).  t0 = bf16(v), t1 = bf16(v - t0), t2 = bf16(v - t0 - t1): each difference is
// exact in fp32, and the three terms add back to v exactly.
__global__ void dl_split_kernel(const float* __restrict__ dl, __nv_bfloat16* __restrict__ out,
                                int N, int E, int Epad) {
  const int64_t n = (int64_t)N * Epad;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / Epad;
    const int e = (int)(i - t * Epad);
    const float v = e < E ? dl[t * E + e] : 0.0f;
    const __nv_bfloat16 a = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(a);
    const __nv_bfloat16 b = __float2bfloat16_rn(r1);
    const __nv_bfloat16 c = __float2bfloat16_rn(r1 - __bfloat162float(b));
    __nv_bfloat16* row = out + t * 3 * Epad;
    row[e] = a;
    row[Epad + e] = b;
    row[2 * Epad + e] = c;
  }
}

// db partials: CTA (x, s) sums experts 32x..32x+31 over token slice s; its 8 warps take
// consecutive runs of the slice, lane = expert, and add their sums in warp order.
__global__ void __launch_bounds__(256)
db_partial_kernel(const float* __restrict__ dl, float* __restrict__ part, int N, int E) {
  __shared__ float red[8][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 32 + lane;
  const int s = blockIdx.y;
  const int t0 = (int)((int64_t)N * s / DB_SLICES), t1 = (int)((int64_t)N * (s + 1) / DB_SLICES);
  const int len = t1 - t0;
  const int a = t0 + (int)((int64_t)len * warp / 8), b = t0 + (int)((int64_t)len * (warp + 1) / 8);
  float acc = 0.0f;
  if (e < E)
    for (int t = a; t < b; ++t) acc += dl[(int64_t)t * E + e];
  red[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && e < E) {
    float v = red[0][lane];
#pragma unroll
    for (int w = 1; w < 8; ++w) v += red[w][lane];
    part[(int64_t)s * E + e] = v;
  }
}

__global__ void db_final_kernel(const float* __restrict__ part, float* __restrict__ db, int E) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  float v = 0.0f;
  for (int s = 0; s < DB_SLICES; ++s) v += part[(int64_t)s * E + e];
  db[e] = v;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// bf16 [rows, cols] row-major, 64 x 64 boxes (MN-major operand tiles), 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)BK};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int epad_of(int E) { return (E + BM - 1) / BM * BM; }

}  // namespace

size_t router_bwd_ws_bytes(const Cfg& c) {
  const size_t Epad = (size_t)epad_of(c.E);
  const size_t split = ((size_t)c.N * 3 * Epad * 2 + 255) & ~size_t(255);
  return split + (size_t)DB_SLICES * c.E * 4;
}

cudaError_t launch_router_dw_tc(const Cfg& c, const float* dlogits, const void* x, float* dw_router,
                                float* db_router, void* ws, int* status, cudaStream_t s) {
  const int Epad = epad_of(c.E);
  __nv_bfloat16* split = static_cast<__nv_bfloat16*>(ws);
  float* part = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                         (((size_t)c.N * 3 * Epad * 2 + 255) & ~size_t(255)));
  const int g = num_sms() * 4;
  dl_split_kernel<<<g, 256, 0, s>>>(dlogits, split, c.N, c.E, Epad);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap ma, mb;
  if (!make_map(&ma, split, 3 * (uint64_t)Epad, c.N) || !make_map(&mb, x, c.d, c.N))
    return cudaErrorInvalidValue;
  static bool attr_set[64];  // function attributes once per device, outside stream capture
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_set[dev & 63]) {
    cudaFuncSetAttribute(router_dw_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)SMEM_BYTES);
    attr_set[dev & 63] = true;
  }
  const int tiles = (Epad / BM) * ((c.d + BN - 1) / BN);
  const int grid = tiles < num_sms() ? tiles : num_sms();
  DwParams p{dw_router, status, c.N, c.E, Epad, c.d};
  router_dw_tc_kernel<<<grid, THREADS, SMEM_BYTES, s>>>(ma, mb, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  db_partial_kernel<<<dim3((c.E + 31) / 32, DB_SLICES), 256, 0, s>>>(dlogits, part, c.N, c.E);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  db_final_kernel<<<(c.E + 255) / 256, 256, 0, s>>>(part, db_router, c.E);
  return cudaGetLastError();
}

}  // namespace moe
