// ffn_tc2.cu -- the grouped SwiGLU expert FFN on pairs of SMs (tcgen05 cta_group::2).
//
// Same computation as ffn_tc.cu (Ultralytics glossary "Expert Parallelism", section
// "How tokens move between GPUs", step 3: every rank runs its local experts on the
// rows it received; fudan-mlsys-cn chapter 10, section 10.5: the shared expert sees
// every token): G1 h = silu(X Wg^T) * (X Wu^T), G2 Y = h Wd^T, bf16 in, fp32 accumulate.
//
// Why pairs: in the single-SM kernel every 128x256x64 block moves 16 KB of token rows
// and 32 KB of weights into one SM's shared memory, and that weight stream (not the
// tensor core, not DRAM) bounds it.  Here two CTAs of a cluster (one TPC) compute a
// 256x256 tile with one tcgen05.mma.cta_group::2 (M=256, N=256, K=16): each CTA loads
// its own 128 token rows and HALF of the weight tile (G1: CTA 0 the 128 gate rows,
// CTA 1 the matching 128 up rows; G2: one 128-row half each), so each SM moves 32 KB
// per block instead of 48.  Each CTA's tensor memory holds its own 128 rows of the
// 256x256 accumulator, and its own epilogue writes them.
//
// Roles (both CTAs run all of them; only the pair's leader, cluster rank 0, issues MMAs):
//   warp 0      TMA producer: loads into this CTA's 6-stage ring; every copy completes
//               on the LEADER's full barrier (cta_group::2 form of the bulk tensor copy),
//               which the leader's producer arms for both CTAs' bytes
//   warp 1      TMEM allocation for the pair (cta_group::2); in the leader, the single
//               MMA-issuing thread, whose commits arrive on the barriers of both CTAs
//               (stage release, accumulator ready, final drain)
//   warps 2-5   epilogue over this CTA's 128 accumulator rows; each warp releases the
//               accumulator on the leader's barrier (a remote arrive from CTA 1)
// Tiles are 256 rows of one segment (an expert's send rows, or the shared expert's
// tokens) x 256 output columns; the pair walks them in the order of the single-SM
// kernel.  Every mbarrier wait is bounded (about 2 s) and reports through the status
// word; the pair meets at cluster barriers after initialisation and before teardown.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128;              // rows per CTA (TMEM lanes)
constexpr int PM = 256;              // rows per pair tile
constexpr int BK = 64;               // K per stage: one 128-byte swizzle row
constexpr int BN = 256;              // accumulator columns per tile (output columns)
constexpr int BH = 128;              // weight rows per CTA per stage (half of BN)
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BH * BK * 2;  // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;
constexpr int MAX_SEG = kMaxExperts + 1;
constexpr uint64_t WAIT_NS = 2000000000ull;

enum { GATE_UP = 0, DOWN = 1 };

// kind::f16, D fp32, A/B bf16 K-major, N = 256, M = 256 (the pair's rows)
constexpr uint32_t IDESC2 = idesc_bf16_f32(PM, BN);

struct Tc2Params {
  const int32_t* expert_start;
  const int32_t* kept_counts;
  __nv_bfloat16* out0;  // routed output, indexed by send-buffer row
  __nv_bfloat16* out1;  // shared-expert output, indexed by token
  __nv_bfloat16* gu0;   // optional (training): g and u of each routed row, [rows, 2F]
  __nv_bfloat16* gu1;   // and of the shared expert, [N, 2Fs]
  int* err;
  int E, n_shared, d, F, Fs;
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

// ---------------------------------------------------------------- pair primitives
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr(p)), "r"(rank));
  return r;
}
// TMA tile copy into this CTA's shared memory; the transaction completes on an
// mbarrier that may live in the peer CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_pair(void* dst, const CUtensorMap* map, uint32_t bar,
                                              int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(saddr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void mma_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive (once in each CTA of the pair) on the mbarrier at this offset when all prior
// tcgen05 operations of this thread have completed.
__device__ __forceinline__ void commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(saddr(bar)),
      "h"((uint16_t)0x3)
      : "memory");
}
__device__ __forceinline__ void arrive_remote(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
               : "memory");
}

// Bounded wait (as in ffn_tc.cu).  False when the wait expired or another role of this
// CTA already gave up.
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

// ---------------------------------------------------------------- tiles
struct Tile {
  int seg, m0, n0, rows, row_base;
};

template <int MODE>
__device__ __forceinline__ int n_tiles(bool routed, const Tc2Params& p) {
  if (MODE == GATE_UP) return ((routed ? p.F : p.Fs) + BN / 2 - 1) / (BN / 2);
  return (p.d + BN - 1) / BN;
}

template <int MODE>
__device__ __forceinline__ Tile decode(const Ctl* ctl, int nseg, int t) {
  int lo = 0, hi = nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ctl->tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  Tile tl;
  tl.seg = lo;
  const int local = t - ctl->tile_start[lo];
  const int mt = ctl->mtiles[lo];
  tl.m0 = (local % mt) * PM;  // column-tile major: concurrent pairs share a weight tile
  tl.n0 = (local / mt) * (MODE == GATE_UP ? BN / 2 : BN);
  tl.rows = ctl->rows[lo];
  tl.row_base = ctl->row_base[lo];
  return tl;
}

// ---------------------------------------------------------------- kernel
template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
grouped_ffn2_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                    Tc2Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + (size_t)STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0: the pair's leader
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int nseg = p.E + (p.n_shared > 0 ? 1 : 0);

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&ctl->tfull[a], 1);
      mbar_init(&ctl->tempty[a], 8);  // 4 epilogue warps in each CTA of the pair
    }
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     saddr(&ctl->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  if (warp == 2) {  // per-segment pair-tile table (identical in both CTAs)
    int base = 0;
    for (int s0 = 0; s0 < nseg; s0 += 32) {
      const int s = s0 + lane;
      int v = 0;
      if (s < nseg) {
        const bool routed = s < p.E;
        const int cnt = routed ? p.kept_counts[s] : p.n_shared;
        const int mt = (cnt + PM - 1) / PM;
        ctl->mtiles[s] = mt > 0 ? mt : 1;
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
  cluster_sync();  // both CTAs' barriers exist before any copy or arrive targets them
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  const int total = ctl->tile_start[nseg];

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = pair; t < total && ok; t += npairs) {
        const Tile tl = decode<MODE>(ctl, nseg, t);
        const bool routed = tl.seg < p.E;
        const int Fx = routed ? p.F : p.Fs;
        const int K = (MODE == GATE_UP) ? p.d : Fx;
        const CUtensorMap* ma = routed ? &tmA0 : &tmA1;
        const CUtensorMap* mb = routed ? &tmB0 : &tmB1;
        const int a_row = tl.row_base + tl.m0 + (int)rank * BM;
        int b_row;
        if (MODE == GATE_UP)  // CTA 0: gate rows n0..n0+127; CTA 1: the matching up rows
          b_row = (routed ? tl.seg * 2 * p.F : 0) + tl.n0 + (int)rank * Fx;
        else
          b_row = (routed ? tl.seg * p.d : 0) + tl.n0 + (int)rank * BH;
        for (int k0 = 0; k0 < K; k0 += BK) {
          if (!mbar_wait(&ctl->empty[stage], phase ^ 1, ctl, p.err, 1)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + (size_t)stage * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          if (rank == 0) mbar_expect_tx(&ctl->full[stage], 2 * STAGE_BYTES);
          const uint32_t lead_full = peer_addr(&ctl->full[stage], 0);
          tma_load_pair(sa, ma, lead_full, k0, a_row);
          tma_load_pair(sb, mb, lead_full, k0, b_row);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (the leader's lane 0)
    if (lane == 0) {
      if (rank == 0) {
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        bool issued = false;
        for (int t = pair; t < total && ok; t += npairs) {
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
            if (!mbar_wait(&ctl->full[stage], phase, ctl, p.err, 3)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = saddr(smem + (size_t)stage * STAGE_BYTES);
            const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              mma_pair(dt, sdesc(a0 + kk * 32), sdesc(b0 + kk * 32), IDESC2,
                       (k0 > 0 || kk > 0) ? 1u : 0u);
            issued = true;
            commit_pair(&ctl->empty[stage]);  // both CTAs may refill this stage
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          commit_pair(&ctl->tfull[acc]);  // both CTAs' accumulator halves are ready
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
        }
        if (issued) commit_pair(&ctl->drain);
      }
      // every MMA writing this CTA's tensor memory has finished before it is freed
      if (pair < total) {
        const uint64_t t0 = now_ns();
        while (!mbar_try_wait(&ctl->drain, 0) && now_ns() - t0 < WAIT_NS) {
        }
      }
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2-5, both CTAs)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;
    const uint32_t lead_tempty0 = peer_addr(&ctl->tempty[0], 0);
    const uint32_t lead_tempty1 = peer_addr(&ctl->tempty[1], 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = pair; t < total; t += npairs) {
      const Tile tl = decode<MODE>(ctl, nseg, t);
      const bool routed = tl.seg < p.E;
      const int ncols = (MODE == GATE_UP) ? (routed ? p.F : p.Fs) : p.d;
      __nv_bfloat16* out = routed ? p.out0 : p.out1;
      const int my_row = tl.m0 + (int)rank * BM + r;  // row within the segment
      const bool valid = my_row < tl.rows;
      if (!mbar_wait(&ctl->tfull[acc], acc_phase, ctl, p.err, 4)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      __nv_bfloat16* orow = out + (int64_t)(tl.row_base + my_row) * ncols;
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
              __nv_bfloat16* gurow = gubase + (int64_t)(tl.row_base + my_row) * (2 * ncols);
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
      if (lane == 0) {  // release this accumulator on the leader's barrier
        if (rank == 0)
          mbar_arrive(&ctl->tempty[acc]);
        else
          arrive_remote(acc ? lead_tempty1 : lead_tempty0);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no copy, MMA or arrive of the pair targets this CTA any more
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
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

template <int MODE>
cudaError_t launch_pair(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
                        const CUtensorMap& b1, const Tc2Params& p, cudaStream_t s) {
  auto k = grouped_ffn2_kernel<MODE>;
  static bool attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_set[dev & 63]) {
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
    attr_set[dev & 63] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(num_sms() & ~1));  // one CTA per SM, whole pairs
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, a0, a1, b0, b1, p);
}

}  // namespace

cudaError_t launch_ffn_tc2(const Cfg& c, const void* xperm, const int32_t* expert_start,
                           const int32_t* kept_counts, const void* w_gate_up, const void* w_down,
                           const void* x, const void* shared_gate_up, const void* shared_down,
                           void* yperm, void* yshared, void* h, int* status, cudaStream_t s,
                           void* gu_save) {
  const bool sh = c.Fs > 0;
  __nv_bfloat16* h_routed = static_cast<__nv_bfloat16*>(h);
  __nv_bfloat16* h_shared = h_routed + (size_t)c.send_rows * c.F;
  __nv_bfloat16* gu_routed = static_cast<__nv_bfloat16*>(gu_save);
  __nv_bfloat16* gu_shared = gu_routed ? gu_routed + (size_t)c.send_rows * 2 * c.F : nullptr;
  CUtensorMap a0, a1, b0, b1;
  // G1: A = send rows [S, d] / tokens [N, d] (128-row boxes); B = [E*2F, d] / [2Fs, d]
  // (128-row boxes: the gate half or the up half)
  if (!make_map(&a0, xperm, c.d, c.send_rows, BM) ||
      !make_map(&b0, w_gate_up, c.d, (uint64_t)c.E * 2 * c.F, BH))
    return cudaErrorInvalidValue;
  a1 = a0;
  b1 = b0;
  if (sh && (!make_map(&a1, x, c.d, c.N, BM) || !make_map(&b1, shared_gate_up, c.d, 2 * c.Fs, BH)))
    return cudaErrorInvalidValue;
  Tc2Params p{expert_start, kept_counts, h_routed, h_shared, gu_routed, sh ? gu_shared : nullptr,
              status, c.E, sh ? c.N : 0, c.d, c.F, c.Fs};
  cudaError_t e = launch_pair<GATE_UP>(a0, a1, b0, b1, p, s);
  if (e != cudaSuccess) return e;
  // G2: A = h [S, F] / [N, Fs]; B = [E*d, F] / [d, Fs] (128-row halves of a 256-row tile)
  if (!make_map(&a0, h_routed, c.F, c.send_rows, BM) ||
      !make_map(&b0, w_down, c.F, (uint64_t)c.E * c.d, BH))
    return cudaErrorInvalidValue;
  a1 = a0;
  b1 = b0;
  if (sh && (!make_map(&a1, h_shared, c.Fs, c.N, BM) || !make_map(&b1, shared_down, c.Fs, c.d, BH)))
    return cudaErrorInvalidValue;
  p.out0 = static_cast<__nv_bfloat16*>(yperm);
  p.out1 = static_cast<__nv_bfloat16*>(yshared);
  p.gu0 = p.gu1 = nullptr;
  return launch_pair<DOWN>(a0, a1, b0, b1, p, s);
}

}  // namespace moe
