// ffn_tc.cu -- grouped SwiGLU expert FFN on the 5th-generation tensor cores (bf16).
//
// Ultralytics glossary "Expert Parallelism", section "How tokens move between GPUs",
// step 3: each rank runs its local experts on the rows it received; every expert is
// a feed-forward block, here SwiGLU: h = silu(X Wg^T) * (X Wu^T), Y = h Wd^T.
// fudan-mlsys-cn chapter 10, section 10.5: a shared expert processes every token.
//
// Two persistent grouped GEMMs, one CTA per SM, each a warp-specialised pipeline:
//   warp 0      TMA producer: A (rows of one expert segment) and B (that expert's
//               weights) K-slices into a 4-stage shared-memory ring (128B swizzle)
//   warp 1      TMEM owner + single-thread tcgen05.mma issuer (M=128, N=256, K=16,
//               bf16 x bf16 -> fp32 in TMEM, two 256-column accumulators)
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, math, bf16 stores
//   G1 (gate_up): B tile = 128 gate rows + the matching 128 up rows, so one
//       accumulator holds both halves and the epilogue writes h = silu(g) * u
//       (bf16) for 128 columns.
//   G2 (down):    B tile = 256 rows of Wd; the epilogue writes Y (bf16).
// Segments: routed expert e owns send-buffer rows [expert_start[e], +kept_counts[e]);
// the shared expert is one more segment over the N token rows.  Tiles never span two
// segments: rows of a 128-row tile past the segment's end are loaded (next segment
// or TMA zero fill) but never stored.  The tile list is built on the device from the
// counts, so nothing returns to the host between dispatch and compute.  Tile order
// inside a segment is column-tile major, row-tile minor: CTAs running at the same
// time share the same weight tile through L2.
//
// Every mbarrier wait is bounded (about 2 s): on expiry the CTA records an error
// code, stops all roles, waits (bounded) for its own TMA copies and MMAs, frees its
// TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128;              // rows per tile (TMEM lanes)
constexpr int BK = 64;               // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int BN = 256;              // accumulator columns per tile
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;
constexpr int MAX_SEG = kMaxExperts + 1;
constexpr uint64_t WAIT_NS = 2000000000ull;

enum { GATE_UP = 0, DOWN = 1 };

constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);

struct TcParams {
  const int32_t* expert_start;
  const int32_t* kept_counts;
  __nv_bfloat16* out0;  // routed output, indexed by send-buffer row
  __nv_bfloat16* out1;  // shared-expert output, indexed by token
  int* err;
  int E, n_shared, d, F, Fs;
  int stall_cta;  // self-test only: this CTA arms its first ring slot without loading it
  __nv_bfloat16* gu0;  // optional (training): g and u of each routed row, [rows, 2F]
  __nv_bfloat16* gu1;  // and of the shared expert, [N, 2Fs]
};

struct Ctl {
  uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], drain;
  uint32_t tmem_base;
  int abort;
  int tile_start[MAX_SEG + 1];
  int mtiles[MAX_SEG];
  int rows[MAX_SEG];
  int row_base[MAX_SEG];
};

constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + sizeof(Ctl);

// Bounded wait.  False when the wait expired (error recorded) or another role
// already gave up.  Waits on another role's progress (ring slot freed, accumulator
// filled or drained) get twice the limit of the MMA issuer's wait for a loaded slot,
// so a copy that never lands is reported as such (code 3), not as a stalled consumer.
__device__ bool mbar_wait(uint64_t* b, uint32_t parity, Ctl* ctl, int* err, int code,
                          uint64_t limit_ns = 2 * WAIT_NS) {
  if (mbar_try_wait(b, parity)) return true;
  const uint64_t t0 = now_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(b, parity)) return true;
    if ((i & 63) == 0) {
      if (*(volatile int*)&ctl->abort) return false;
      if (now_ns() - t0 > limit_ns) {
        *(volatile int*)&ctl->abort = 1;
        atomicExch(err, code);
        return false;
      }
    }
  }
}
// ---------------------------------------------------------------- tiles
struct Tile {
  int seg, m0, n0, rows, row_base;
};

template <int MODE>
__device__ __forceinline__ int n_tiles(bool routed, const TcParams& p) {
  if (MODE == GATE_UP) return ((routed ? p.F : p.Fs) + BN / 2 - 1) / (BN / 2);
  return (p.d + BN - 1) / BN;
}

template <int MODE>
__device__ __forceinline__ Tile decode(const Ctl* ctl, int nseg, int t) {
  int lo = 0, hi = nseg - 1;  // last segment whose first tile is <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ctl->tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  Tile tl;
  tl.seg = lo;
  const int local = t - ctl->tile_start[lo];
  const int mt = ctl->mtiles[lo];
  tl.m0 = (local % mt) * BM;
  tl.n0 = (local / mt) * (MODE == GATE_UP ? BN / 2 : BN);
  tl.rows = min(BM, ctl->rows[lo] - tl.m0);
  tl.row_base = ctl->row_base[lo];
  return tl;
}

// TMA coordinates of one tile: A rows (segment rows), B rows (weights), K extent.
struct Loads {
  bool routed;
  int K, a_row, b_row, b_row2;
};

template <int MODE>
__device__ __forceinline__ Loads loads(const Tile& tl, const TcParams& p) {
  Loads l;
  l.routed = tl.seg < p.E;
  const int Fx = l.routed ? p.F : p.Fs;
  l.K = (MODE == GATE_UP) ? p.d : Fx;
  l.a_row = tl.row_base + tl.m0;
  if (MODE == GATE_UP) {
    l.b_row = (l.routed ? tl.seg * 2 * p.F : 0) + tl.n0;
    l.b_row2 = l.b_row + Fx;
  } else {
    l.b_row = (l.routed ? tl.seg * p.d : 0) + tl.n0;
    l.b_row2 = 0;
  }
  return l;
}

// ---------------------------------------------------------------- kernel
template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
grouped_ffn_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                   const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                   TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + (size_t)STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nseg = p.E + (p.n_shared > 0 ? 1 : 0);

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&ctl->tfull[a], 1);
      mbar_init(&ctl->tempty[a], 4);
    }
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA0)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB0)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     saddr(&ctl->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (warp == 2) {  // per-segment tile table
    int base = 0;
    for (int s0 = 0; s0 < nseg; s0 += 32) {
      const int s = s0 + lane;
      int v = 0;
      if (s < nseg) {
        const bool routed = s < p.E;
        const int cnt = routed ? p.kept_counts[s] : p.n_shared;
        const int mt = (cnt + BM - 1) / BM;
        ctl->mtiles[s] = mt;
        ctl->rows[s] = cnt;
        ctl->row_base[s] = routed ? p.expert_start[s] : 0;
        v = mt * n_tiles<MODE>(routed, p);
      }
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      if (s < nseg) ctl->tile_start[s] = base + incl - v;
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) ctl->tile_start[nseg] = base;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  const int total = ctl->tile_start[nseg];

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;  // per-stage bits, for the abort drain
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Loads ld = loads<MODE>(decode<MODE>(ctl, nseg, t), p);
        const CUtensorMap* ma = ld.routed ? &tmA0 : &tmA1;
        const CUtensorMap* mb = ld.routed ? &tmB0 : &tmB1;
        for (int k0 = 0; k0 < ld.K; k0 += BK) {
          if (!mbar_wait(&ctl->empty[stage], phase ^ 1, ctl, p.err, 1)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + (size_t)stage * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          mbar_expect_tx(&ctl->full[stage], STAGE_BYTES);
          if (blockIdx.x == p.stall_cta && t == (int)blockIdx.x && k0 == 0) {
            // self-test: the slot's bytes never arrive, so the MMA's bounded wait runs out
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
            continue;
          }
          tma_load(sa, ma, &ctl->full[stage], k0, ld.a_row);
          if (MODE == GATE_UP) {
            tma_load(sb, mb, &ctl->full[stage], k0, ld.b_row);
            tma_load(sb + B_BYTES / 2, mb, &ctl->full[stage], k0, ld.b_row2);
          } else {
            tma_load(sb, mb, &ctl->full[stage], k0, ld.b_row);
          }
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
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool issued = false;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile tl = decode<MODE>(ctl, nseg, t);
        const bool routed = tl.seg < p.E;
        const int K = (MODE == GATE_UP) ? p.d : (routed ? p.F : p.Fs);
        if (!mbar_wait(&ctl->tempty[acc], acc_phase ^ 1, ctl, p.err, 2)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dt = tmem_base + (uint32_t)(acc * BN);
        for (int k0 = 0; k0 < K; k0 += BK) {
          if (!mbar_wait(&ctl->full[stage], phase, ctl, p.err, 3, WAIT_NS)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = saddr(smem + (size_t)stage * STAGE_BYTES);
          const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma(dt, sdesc(a0 + kk * 32), sdesc(b0 + kk * 32), IDESC, (k0 > 0 || kk > 0) ? 1u : 0u);
          issued = true;
          tc_commit(&ctl->empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(&ctl->tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
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
    const int r = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = decode<MODE>(ctl, nseg, t);
      const bool routed = tl.seg < p.E;
      const int ncols = (MODE == GATE_UP) ? (routed ? p.F : p.Fs) : p.d;
      __nv_bfloat16* out = routed ? p.out0 : p.out1;
      const bool valid = r < tl.rows;
      if (!mbar_wait(&ctl->tfull[acc], acc_phase, ctl, p.err, 4)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      __nv_bfloat16* orow = out + (int64_t)(tl.row_base + tl.m0 + r) * ncols;
      if (MODE == GATE_UP) {
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(tb + c, g);
          tmem_ld32(tb + BN / 2 + c, u);
          tmem_ld_wait(g);
          tmem_ld_wait(u);
          if (valid) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
              const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
              const float h0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
              const float h1 = __fdividef(g1, 1.0f + __expf(-g1)) * u1;
              pk[i] = pack_bf16(h0, h1);
            }
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int col = tl.n0 + c + v * 8;
              if (col < ncols)
                *reinterpret_cast<uint4*>(orow + col) =
                    make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
            __nv_bfloat16* gubase = routed ? p.gu0 : p.gu1;
            if (gubase) {  // training: keep g and u for the backward pass
              __nv_bfloat16* gurow = gubase + (int64_t)(tl.row_base + tl.m0 + r) * (2 * ncols);
              uint32_t pg[16], pu[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                pg[i] = pack_bf16(__uint_as_float(g[2 * i]), __uint_as_float(g[2 * i + 1]));
                pu[i] = pack_bf16(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1]));
              }
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const int col = tl.n0 + c + v * 8;
                if (col < ncols) {
                  *reinterpret_cast<uint4*>(gurow + col) =
                      make_uint4(pg[4 * v], pg[4 * v + 1], pg[4 * v + 2], pg[4 * v + 3]);
                  *reinterpret_cast<uint4*>(gurow + ncols + col) =
                      make_uint4(pu[4 * v], pu[4 * v + 1], pu[4 * v + 2], pu[4 * v + 3]);
                }
              }
            }
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t y[32];
          tmem_ld32(tb + c, y);
          tmem_ld_wait(y);
          if (valid) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16(__uint_as_float(y[2 * i]), __uint_as_float(y[2 * i + 1]));
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int col = tl.n0 + c + v * 8;
              if (col < ncols)
                *reinterpret_cast<uint4*>(orow + col) =
                    make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// ---------------------------------------------------------------- host side
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

// 2-D bf16 map over a row-major [rows, K] matrix; box = 64 K-elements x box_rows.
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

cudaError_t launch_ffn_tc(const Cfg& c, const void* xperm, const int32_t* expert_start,
                          const int32_t* kept_counts, const void* w_gate_up, const void* w_down,
                          const void* x, const void* shared_gate_up, const void* shared_down,
                          void* yperm, void* yshared, void* h, int* status, cudaStream_t s,
                          int stall_cta, void* gu_save) {
  const bool sh = c.Fs > 0;
  __nv_bfloat16* h_routed = static_cast<__nv_bfloat16*>(h);
  __nv_bfloat16* h_shared = h_routed + (size_t)c.send_rows * c.F;
  CUtensorMap a0, a1, b0, b1;
  // G1: A = send buffer [A, d] / tokens [N, d]; B = [E*2F, d] / [2Fs, d]
  if (!make_map(&a0, xperm, c.d, c.send_rows, BM) || !make_map(&b0, w_gate_up, c.d, (uint64_t)c.E * 2 * c.F, BN / 2))
    return cudaErrorInvalidValue;
  a1 = a0;
  b1 = b0;
  if (sh && (!make_map(&a1, x, c.d, c.N, BM) || !make_map(&b1, shared_gate_up, c.d, 2 * c.Fs, BN / 2)))
    return cudaErrorInvalidValue;
  __nv_bfloat16* gu_routed = static_cast<__nv_bfloat16*>(gu_save);
  __nv_bfloat16* gu_shared = gu_routed ? gu_routed + (size_t)c.send_rows * 2 * c.F : nullptr;
  TcParams p{expert_start, kept_counts, h_routed, h_shared, status,
             c.E, sh ? c.N : 0, c.d, c.F, c.Fs, stall_cta, gu_routed, sh ? gu_shared : nullptr};
  const int grid = num_sms();
  auto k1 = grouped_ffn_kernel<GATE_UP>;
  auto k2 = grouped_ffn_kernel<DOWN>;
  static bool attr_set[64];  // function attributes once per device, outside stream capture
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_set[dev & 63]) {
    cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    attr_set[dev & 63] = true;
  }
  k1<<<grid, THREADS, SMEM_BYTES, s>>>(a0, a1, b0, b1, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // G2: A = h [A, F] / [N, Fs]; B = [E*d, F] / [d, Fs]
  if (!make_map(&a0, h_routed, c.F, c.send_rows, BM) || !make_map(&b0, w_down, c.F, (uint64_t)c.E * c.d, BN))
    return cudaErrorInvalidValue;
  a1 = a0;
  b1 = b0;
  if (sh && (!make_map(&a1, h_shared, c.Fs, c.N, BM) || !make_map(&b1, shared_down, c.Fs, c.d, BN)))
    return cudaErrorInvalidValue;
  p.out0 = static_cast<__nv_bfloat16*>(yperm);
  p.out1 = static_cast<__nv_bfloat16*>(yshared);
  p.stall_cta = -1;  // only the first GEMM takes part in the self-test
  p.gu0 = p.gu1 = nullptr;
  k2<<<grid, THREADS, SMEM_BYTES, s>>>(a0, a1, b0, b1, p);
  return cudaGetLastError();
}

}  // namespace moe
