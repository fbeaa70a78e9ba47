// router_tc.cu -- router logits on the tensor cores for bf16 hidden states.
//
// Ultralytics glossary "Expert Parallelism", section "How tokens move between GPUs",
// step 1: the router is a linear layer that scores every token against every
// expert.  The router weight is fp32 and the logits must be fp32-accurate, while
// the tensor cores multiply bf16.  Since x is already bf16, the weight is split
// into three bf16 terms W = W0 + W1 + W2 (W0 = bf16(W), W1 = bf16(W - W0),
// W2 = bf16(W - W0 - W1); both differences are exact in fp32), every product
// x * Ws is exact in the fp32 accumulator, and what is left out is about 2^-27 |W|.
// When 3 * Epad fits one MMA's N (<= 256, i.e. up to 64 experts) the three terms are
// stacked along N: Ws is [3*Epad, dpad] and each K block of x meets all three terms
// in one MMA, into three column ranges of the accumulator that the epilogue adds; x is
// read once.  Otherwise they are stacked along K: Ws is [Epad, 3*dpad], one GEMM with
// K' = 3 * dpad computes x . W0^T + x . W1^T + x . W2^T with the x K-coordinate
// wrapping modulo dpad (x read three times).
//
//   split_kernel   W [E, d] fp32 -> Ws (either layout) bf16 (zero padded)
//   router_gemm    one CTA per (128-token tile, K' slice): TMA -> 4-stage ring ->
//                  tcgen05.mma (M=128, N=Epad) -> TMEM -> fp32 partial logits
// Slices ("split-K") put all SMs to work when there are few token tiles; the
// selection kernel (route.cu) adds the slices in a fixed order plus the bias.
//
// Accumulation length: the tensor core adds each MMA's products into the fp32
// accumulator with a rounding that drops bits toward zero, so the error of one
// accumulation chain grows with its number of MMA steps (at K' = 21504 the logits
// came out about 1.7e-5 low in relative terms).  Each CTA therefore spreads its K
// blocks round-robin over n_acc TMEM accumulators, the slicing keeps every chain at
// or below kChainK elements, and the chains are summed in round-to-nearest fp32
// (epilogue, then the selection kernel) in a fixed order.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128, BK = 64, STAGES = 4, THREADS = 192;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_MAX_BYTES = 256 * BK * 2;       // 32 KB (Epad <= 256)
constexpr int STAGE_BYTES = A_BYTES + B_MAX_BYTES;
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr int kChainK = 4096;  // longest K per accumulation chain (elements)

struct RCtl {
  uint64_t full[STAGES], empty[STAGES], tfull, drain;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + sizeof(RCtl);

struct RParams {
  float* partial;  // [nsplit][N][Epad]
  int* err;
  int N, Epad, nkb_d, kb_per_split, total_kb, n_acc, acc_cols;
  int terms_n;  // term column ranges per accumulator (3 when stacked along N, else 1)
  uint32_t idesc, tmem_cols, b_bytes;
};

__device__ bool wait_bar(uint64_t* b, uint32_t parity, RCtl* ctl, int* err, int code) {
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

__global__ void split_kernel(const float* __restrict__ W, __nv_bfloat16* __restrict__ Ws, int E,
                             int d, int Epad, int dpad, int stacked_n) {
  const int64_t total = (int64_t)Epad * dpad;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int e = (int)(i / dpad), c = (int)(i % dpad);
    const float w = (e < E && c < d) ? W[(int64_t)e * d + c] : 0.0f;
    const __nv_bfloat16 w0 = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(w0);
    const __nv_bfloat16 w1 = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(w1);
    if (stacked_n) {  // term t of expert e is row t * Epad + e of [3*Epad, dpad]
      Ws[(int64_t)e * dpad + c] = w0;
      Ws[((int64_t)Epad + e) * dpad + c] = w1;
      Ws[((int64_t)2 * Epad + e) * dpad + c] = __float2bfloat16_rn(r2);
    } else {          // term t at columns t * dpad of row e of [Epad, 3*dpad]
      __nv_bfloat16* row = Ws + (int64_t)e * 3 * dpad;
      row[c] = w0;
      row[dpad + c] = w1;
      row[2 * dpad + c] = __float2bfloat16_rn(r2);
    }
  }
}

__global__ void __launch_bounds__(THREADS, 1)
router_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   RParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  RCtl* ctl = reinterpret_cast<RCtl*>(smem + (size_t)STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * BM;
  const int kb0 = blockIdx.y * p.kb_per_split;
  const int kb1 = min(kb0 + p.kb_per_split, p.total_kb);
  const uint32_t b_bytes = p.b_bytes;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    mbar_init(&ctl->tfull, 1);
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(&ctl->tmem_base, p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_bar(&ctl->empty[stage], phase ^ 1, ctl, p.err, 11)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem + (size_t)stage * STAGE_BYTES;
        mbar_expect_tx(&ctl->full[stage], A_BYTES + b_bytes);
        tma_load(sa, &tmX, &ctl->full[stage], (kb % p.nkb_d) * BK, m0);
        tma_load(sa + A_BYTES, &tmW, &ctl->full[stage], kb * BK, 0);
        armed |= 1u << stage;
        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) {
        const uint64_t t0 = now_ns();
        for (int s = 0; s < STAGES; ++s)
          if (armed >> s & 1u)
            while (!mbar_try_wait(&ctl->full[s], armed_parity >> s & 1u) &&
                   now_ns() - t0 < WAIT_NS) {
            }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true, issued = false;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_bar(&ctl->full[stage], phase, ctl, p.err, 12)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = saddr(smem + (size_t)stage * STAGE_BYTES);
        const uint32_t b0 = a0 + A_BYTES;
        const int j = kb - kb0;  // K blocks go round-robin over the accumulators
        const uint32_t dt = tmem_base + (uint32_t)((j % p.n_acc) * p.acc_cols);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc_mma(dt, sdesc(a0 + kk * 32), sdesc(b0 + kk * 32), p.idesc,
                 (j >= p.n_acc || kk > 0) ? 1u : 0u);
        issued = true;
        tc_commit(&ctl->empty[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (ok && issued) tc_commit(&ctl->tfull);
      if (issued) {
        tc_commit(&ctl->drain);
        const uint64_t t0 = now_ns();
        while (!mbar_try_wait(&ctl->drain, 0) && now_ns() - t0 < WAIT_NS) {
        }
      }
    }
  } else {  // epilogue: fp32 partial logits, one token row per thread
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int row = m0 + r;
    if (kb1 > kb0 && wait_bar(&ctl->tfull, 0, ctl, p.err, 13)) {
      tc_fence_after();
      float* out = p.partial + ((int64_t)blockIdx.y * p.N + row) * p.Epad;
      const int n_used = min(p.n_acc, kb1 - kb0);
      const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
      for (int c = 0; c < p.Epad; c += 32) {
        uint32_t v[32];
        tmem_ld32(lane_base + (uint32_t)c, v);
        tmem_ld_wait(v);
        // fixed-order round-to-nearest sum over the term ranges, then the accumulators
        for (int tm = 0; tm < p.terms_n; ++tm) {
          for (int a = (tm == 0 ? 1 : 0); a < n_used; ++a) {
            uint32_t u[32];
            tmem_ld32(lane_base + (uint32_t)(a * p.acc_cols + tm * p.Epad + c), u);
            tmem_ld_wait(u);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              v[i] = __float_as_uint(__fadd_rn(__uint_as_float(v[i]), __uint_as_float(u[i])));
          }
        }
        if (row < p.N) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<uint4*>(out + c + 4 * i) =
                make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
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

bool make_map(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {K, rows};
  const cuuint64_t strides[1] = {K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

RouterPlan router_plan(const Cfg& c) {
  RouterPlan rp;
  rp.Epad = (c.E + 31) / 32 * 32;
  rp.dpad = (c.d + BK - 1) / BK * BK;
  rp.stacked_n = 3 * rp.Epad <= 256 ? 1 : 0;
  const int ncols = rp.stacked_n ? 3 * rp.Epad : rp.Epad;  // MMA N
  rp.acc_cols = 32;
  while (rp.acc_cols < ncols) rp.acc_cols <<= 1;
  rp.n_acc = 512 / rp.acc_cols;
  if (rp.n_acc > 4) rp.n_acc = 4;
  const int tiles = (c.N + BM - 1) / BM;
  const int total_kb = (rp.stacked_n ? 1 : 3) * (rp.dpad / BK);
  int ns = kSmTarget / tiles;                   // fill the GPU when tiles are few
  if (ns > 16) ns = 16;
  const int chains = (total_kb * BK + kChainK - 1) / kChainK;
  const int ns_prec = (chains + rp.n_acc - 1) / rp.n_acc;  // every chain <= kChainK
  if (ns < ns_prec) ns = ns_prec;
  if (ns < 1) ns = 1;
  if (ns > total_kb) ns = total_kb;
  rp.kb_per_split = (total_kb + ns - 1) / ns;
  rp.nsplit = (total_kb + rp.kb_per_split - 1) / rp.kb_per_split;
  rp.ws_bytes = (size_t)rp.Epad * 3 * rp.dpad * 2;
  rp.partial_bytes = (size_t)rp.nsplit * c.N * rp.Epad * 4;
  return rp;
}

cudaError_t launch_router_gemm(const Cfg& c, const RouterPlan& rp, const void* x,
                               const float* w_router, void* ws_split, float* partial, int* status,
                               cudaStream_t s) {
  __nv_bfloat16* Ws = static_cast<__nv_bfloat16*>(ws_split);
  const int64_t n_el = (int64_t)rp.Epad * rp.dpad;
  int sgrid = (int)((n_el + 255) / 256);
  if (sgrid > num_sms() * 8) sgrid = num_sms() * 8;
  split_kernel<<<sgrid, 256, 0, s>>>(w_router, Ws, c.E, c.d, rp.Epad, rp.dpad, rp.stacked_n);
  CUtensorMap mx, mw;
  const bool ok = rp.stacked_n
                      ? make_map(&mw, Ws, (uint64_t)rp.dpad, 3 * rp.Epad, (uint32_t)(3 * rp.Epad))
                      : make_map(&mw, Ws, (uint64_t)3 * rp.dpad, rp.Epad, (uint32_t)rp.Epad);
  if (!ok || !make_map(&mx, x, c.d, c.N, BM)) return cudaErrorInvalidValue;
  RParams p;
  p.partial = partial;
  p.err = status;
  p.N = c.N;
  p.Epad = rp.Epad;
  p.nkb_d = rp.dpad / BK;
  p.kb_per_split = rp.kb_per_split;
  p.total_kb = (rp.stacked_n ? 1 : 3) * p.nkb_d;
  p.terms_n = rp.stacked_n ? 3 : 1;
  const int ncols = rp.stacked_n ? 3 * rp.Epad : rp.Epad;
  p.idesc = idesc_bf16_f32(BM, ncols);
  p.b_bytes = (uint32_t)ncols * BK * 2;
  p.n_acc = rp.n_acc;
  p.acc_cols = rp.acc_cols;
  uint32_t cols = 32;
  while ((int)cols < rp.n_acc * rp.acc_cols) cols <<= 1;
  p.tmem_cols = cols;
  static bool attr_set[64];  // once per device, outside any stream capture
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_set[dev & 63]) {
    cudaFuncSetAttribute(router_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)SMEM_BYTES);
    attr_set[dev & 63] = true;
  }
  const dim3 grid((c.N + BM - 1) / BM, rp.nsplit);
  router_gemm_kernel<<<grid, THREADS, SMEM_BYTES, s>>>(mx, mw, p);
  return cudaGetLastError();
}

}  // namespace moe
