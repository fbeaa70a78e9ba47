// ffn_tc_small.cu -- grouped SwiGLU expert FFN for segments of few rows (decode).
//
// Ultralytics glossary "Expert Parallelism", section "How tokens move between GPUs",
// step 3: each rank runs its local experts on the rows it received (SwiGLU experts,
// h = silu(X Wg^T) * (X Wu^T), Y = h Wd^T; fudan-mlsys-cn 10.5: shared expert).
//
// When the send buffer holds only a few rows per expert (decoding a handful of
// tokens), a 128-row token tile is mostly padding and the step is a stream over
// the touched experts' weights.  This variant puts a 128-row weight slab on the MMA's
// M side and the segment's tokens on its N side:
//   D[128 weight rows][n] = W_slab . X_rows^T,  n = segment rows in the tile rounded
//   up to 16 (at most 32 rows per tile; longer segments take several tiles),
// and loads tokens in 32-row pieces, so a K step moves 16 KB of weights plus 4 KB of
// tokens instead of 48 KB.  Per CTA (192 threads, persistent, one per SM): warp 0 TMA
// producer (10-stage ring: the bytes in flight set the streaming rate), warp 1 TMEM
// owner and MMA issuer,
// warps 2-5 epilogue.  G1 slab = 64 gate rows + the matching 64 up rows (TMEM lanes
// 0-63 / 64-127, paired through a small shared-memory exchange); G2 slab = 112 rows
// of Wd.  Each epilogue thread owns one feature and writes it for 32 tokens at a
// time.  The down kernel is launched as a programmatic dependent of the gate_up
// kernel: its CTAs start on the SMs that gate_up CTAs leave, set up, and load their
// first weight slices before waiting (griddepcontrol.wait) for the gate_up kernel to
// complete; only then are h rows loaded.  Every mbarrier wait is bounded (about 2 s,
// error code in the status word).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

#ifndef MOE_SMALL_BR
#define MOE_SMALL_BR 32
#endif
#ifndef MOE_SMALL_STAGES
#define MOE_SMALL_STAGES 10
#endif
constexpr int BW = 128;               // weight rows per tile (MMA M, TMEM lanes)
// Down slabs load 112 weight rows (the MMA still computes 128; TMEM lanes 112-127 are
// not written out).  A 7168-wide output then splits into 64 slabs per expert instead
// of 56, which spreads a one-token batch's 9 x 64 tiles over 148 SMs in 3.9 rounds
// instead of 9 x 56 in 3.4 (4 with a mostly idle last one).
constexpr int BW2 = 112;
constexpr int BR = MOE_SMALL_BR;      // token rows per tile (MMA N upper bound)
constexpr int BK = 64;                // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int STAGES = MOE_SMALL_STAGES;  // deep ring: the step streams weights from DRAM
constexpr int PIECE = 32;             // token rows per TMA load
static_assert(BR >= PIECE && BR % PIECE == 0 && BR <= 256, "token tile: whole 32-row pieces");
constexpr int PIECE_BYTES = PIECE * BK * 2;
constexpr int A_BYTES = BW * BK * 2;  // 16 KB weight slab slice (smem room per stage)
constexpr int B_BYTES = BR * BK * 2;  // token rows slice
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr int TMEM_COLS = (2 * BR < 32) ? 32 : 2 * BR;  // two accumulators
constexpr int MAX_SEG = kMaxExperts + 1;
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr int EPI_BAR = 1;            // named barrier of the 4 epilogue warps

enum { GATE_UP = 0, DOWN = 1 };

struct TcParams {
  const int32_t* expert_start;
  const int32_t* kept_counts;
  __nv_bfloat16* out0;  // routed output, indexed by send-buffer row
  __nv_bfloat16* out1;  // shared-expert output, indexed by token
  int* err;
  int E, n_shared, d, F, Fs;
};

struct Ctl {
  uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], drain;
  uint32_t tmem_base;
  int abort;
  int tile_start[MAX_SEG + 1];
  int rtiles[MAX_SEG];
  int rows[MAX_SEG];
  int row_base[MAX_SEG];
  float xchg_g[64][17];  // G1 epilogue: gate values of tokens 16-31 of a chunk
  float xchg_u[64][17];  // G1 epilogue: up values of tokens 0-15 of a chunk
};

constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + sizeof(Ctl);

// Bounded wait.  False when the wait expired (error recorded) or another role
// already gave up.
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

__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(EPI_BAR), "n"(128) : "memory");
}
// Same barrier, returning how many of the 128 epilogue threads passed pred = true.
__device__ __forceinline__ uint32_t epi_count(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.popc.u32 %0, %2, %3, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(EPI_BAR), "n"(128)
      : "memory");
  return r;
}

// ---------------------------------------------------------------- tiles
// Features covered by one slab: G1 64 h-features (64 gate + 64 up weight rows),
// G2 128 output features.
template <int MODE>
__host__ __device__ constexpr int feat_per_tile() {
  return MODE == GATE_UP ? BW / 2 : BW2;
}

template <int MODE>
__device__ __forceinline__ int n_slabs(bool routed, const TcParams& p) {
  const int nf = (MODE == GATE_UP) ? (routed ? p.F : p.Fs) : p.d;
  return (nf + feat_per_tile<MODE>() - 1) / feat_per_tile<MODE>();
}

struct Tile {
  bool routed;
  int seg, r0, f0, rows, row_base, n_pad, pieces, K;
  int w_row, w_row2;  // weight rows of the slab (G1: gate part, up part)
};

template <int MODE>
__device__ __forceinline__ Tile decode(const Ctl* ctl, int nseg, int t, const TcParams& p) {
  int lo = 0, hi = nseg - 1;  // last segment whose first tile is <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ctl->tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  Tile tl;
  tl.seg = lo;
  tl.routed = lo < p.E;
  const int local = t - ctl->tile_start[lo];
  const int rt = ctl->rtiles[lo];
  tl.r0 = (local % rt) * BR;
  tl.f0 = (local / rt) * feat_per_tile<MODE>();
  tl.rows = min(BR, ctl->rows[lo] - tl.r0);
  tl.n_pad = (tl.rows + 15) & ~15;
  tl.pieces = (tl.rows + PIECE - 1) / PIECE;
  tl.row_base = ctl->row_base[lo];
  const int Fx = tl.routed ? p.F : p.Fs;
  tl.K = (MODE == GATE_UP) ? p.d : Fx;
  if (MODE == GATE_UP) {
    tl.w_row = (tl.routed ? tl.seg * 2 * p.F : 0) + tl.f0;
    tl.w_row2 = tl.w_row + Fx;
  } else {
    tl.w_row = (tl.routed ? tl.seg * p.d : 0) + tl.f0;
    tl.w_row2 = 0;
  }
  return tl;
}

// ---------------------------------------------------------------- kernel
// tmW0 / tmW1: routed / shared weights; tmX0 / tmX1: routed / shared token rows
// (32-row boxes).
template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
grouped_ffn_small_kernel(const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmW1,
                   const __grid_constant__ CUtensorMap tmX0, const __grid_constant__ CUtensorMap tmX1,
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
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW0)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX0)) : "memory");
  }
  if (warp == 1) tmem_alloc(&ctl->tmem_base, TMEM_COLS);
  if (warp == 2) {  // per-segment tile table
    // every segment's count and start requested at once (one memory latency), then
    // the prefix over segments 32 at a time
    constexpr int CH = (MAX_SEG + 31) / 32;
    int cnt_r[CH], start_r[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int s = c * 32 + lane;
      cnt_r[c] = s < p.E ? p.kept_counts[s] : (s == p.E ? p.n_shared : 0);
      start_r[c] = s < p.E ? p.expert_start[s] : 0;
    }
    int base = 0;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int s0 = c * 32;
      if (s0 >= nseg) break;
      const int s = s0 + lane;
      int v = 0;
      if (s < nseg) {
        const bool routed = s < p.E;
        const int cnt = cnt_r[c];
        const int rt = (cnt + BR - 1) / BR;
        ctl->rtiles[s] = rt;
        ctl->rows[s] = cnt;
        ctl->row_base[s] = start_r[c];
        v = rt * n_slabs<MODE>(routed, p);
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
  // the down kernel may be scheduled onto SMs this kernel leaves
  if (MODE == GATE_UP) pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;  // per-stage bits, for the abort drain
      bool ok = true;
      // down kernel: h comes from the gate_up kernel, whose tail this kernel may overlap
      // (programmatic launch).  The first tile's weight slices go out for a full ring
      // at once; its h rows follow griddepcontrol.wait (the gate_up kernel has then
      // completed and its writes are visible).
      bool h_ready = MODE == GATE_UP;
      int npend = 0;  // K steps of the first tile armed without their rows (slots 0..)
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile tl = decode<MODE>(ctl, nseg, t, p);
        const CUtensorMap* mw = tl.routed ? &tmW0 : &tmW1;
        const CUtensorMap* mx = tl.routed ? &tmX0 : &tmX1;
        const int x_row = tl.row_base + tl.r0;
        const uint32_t bytes = (MODE == GATE_UP ? A_BYTES : BW2 * BK * 2) + tl.pieces * PIECE_BYTES;
        auto load_rows = [&](int st, int k) {
          uint8_t* sb = smem + (size_t)st * STAGE_BYTES + A_BYTES;
          for (int i = 0; i < tl.pieces; ++i)
            tma_load(sb + i * PIECE_BYTES, mx, &ctl->full[st], k, x_row + i * PIECE);
        };
        for (int k0 = 0; k0 < tl.K; k0 += BK) {
          if (!mbar_wait(&ctl->empty[stage], phase ^ 1, ctl, p.err, 1)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + (size_t)stage * STAGE_BYTES;
          mbar_expect_tx(&ctl->full[stage], bytes);
          if (MODE == GATE_UP) {
            tma_load(sa, mw, &ctl->full[stage], k0, tl.w_row);
            tma_load(sa + A_BYTES / 2, mw, &ctl->full[stage], k0, tl.w_row2);
          } else {
            tma_load(sa, mw, &ctl->full[stage], k0, tl.w_row);
          }
          if (h_ready) load_rows(stage, k0);
          else ++npend;
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
          if (!h_ready && (npend == STAGES || k0 + BK >= tl.K)) {
            pdl_wait();
            asm volatile("fence.proxy.async.global;" ::: "memory");  // h is read by TMA
            for (int j = 0; j < npend; ++j) load_rows(j, j * BK);
            h_ready = true;
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
        const Tile tl = decode<MODE>(ctl, nseg, t, p);
        const uint32_t idesc = idesc_bf16_f32(BW, tl.n_pad);
        if (!mbar_wait(&ctl->tempty[acc], acc_phase ^ 1, ctl, p.err, 2)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dt = tmem_base + (uint32_t)(acc * BR);
        for (int k0 = 0; k0 < tl.K; k0 += BK) {
          if (!mbar_wait(&ctl->full[stage], phase, ctl, p.err, 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = saddr(smem + (size_t)stage * STAGE_BYTES);
          const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma(dt, sdesc(a0 + kk * 32), sdesc(b0 + kk * 32), idesc,
                   (k0 > 0 || kk > 0) ? 1u : 0u);
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
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int lrow = q * 32 + lane;  // slab row held by this thread
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = decode<MODE>(ctl, nseg, t, p);
      // the four warps meet at named barriers below, so they leave together
      const bool ready = mbar_wait(&ctl->tfull[acc], acc_phase, ctl, p.err, 4);
      if (epi_count(ready) != 128) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BR);
      __nv_bfloat16* out = tl.routed ? p.out0 : p.out1;
      const int64_t row0 = (int64_t)tl.row_base + tl.r0;
      if (MODE == GATE_UP) {
        // lanes f (gate) and f + 64 (up) hold the two halves of h feature f0 + f; per
        // 32-token chunk the gate lane finishes tokens 0-15 and the up lane 16-31,
        // after trading the other half through shared memory
        const int F = tl.routed ? p.F : p.Fs;
        const bool gate = q < 2;
        const int fl = lrow & 63;
        const int f = tl.f0 + fl;
        for (int c = 0; c < tl.n_pad; c += 32) {
          uint32_t v[32];
          tmem_ld32(tb + (uint32_t)c, v);
          tmem_ld_wait(v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (gate) ctl->xchg_g[fl][j] = __uint_as_float(v[16 + j]);
            else ctl->xchg_u[fl][j] = __uint_as_float(v[j]);
          }
          epi_sync();
          if (f < F) {
            const int j0 = gate ? 0 : 16;
            const int nj = min(16, tl.rows - c - j0);
            __nv_bfloat16* o = out + (row0 + c + j0) * F + f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (j < nj) {
                const float g = gate ? __uint_as_float(v[j]) : ctl->xchg_g[fl][j];
                const float u = gate ? ctl->xchg_u[fl][j] : __uint_as_float(v[16 + j]);
                o[(int64_t)j * F] = __float2bfloat16_rn(__fdividef(g, 1.0f + __expf(-g)) * u);
              }
            }
          }
          epi_sync();
        }
      } else {
        const int f = tl.f0 + lrow;  // output feature of this lane
        for (int c = 0; c < tl.n_pad; c += 32) {
          uint32_t v[32];
          tmem_ld32(tb + (uint32_t)c, v);
          tmem_ld_wait(v);
          if (lrow < BW2 && f < p.d) {
            const int nj = min(32, tl.rows - c);
            __nv_bfloat16* o = out + (row0 + c) * p.d + f;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nj) o[(int64_t)j * p.d] = __float2bfloat16_rn(__uint_as_float(v[j]));
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
    tmem_dealloc(tmem_base, TMEM_COLS);
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
cudaError_t launch(const CUtensorMap& w0, const CUtensorMap& w1, const CUtensorMap& x0,
                   const CUtensorMap& x1, const TcParams& p, cudaStream_t s) {
  auto kern = grouped_ffn_small_kernel<MODE>;
  static bool attr_set[64];  // once per device, outside any stream capture
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_set[dev & 63]) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    attr_set[dev & 63] = true;
  }
  if (MODE == GATE_UP) {
    kern<<<num_sms(), THREADS, SMEM_BYTES, s>>>(w0, w1, x0, x1, p);
    return cudaGetLastError();
  }
  // the down kernel is a programmatic dependent of the gate_up kernel just before it
  return launch_dependent(kern, dim3(num_sms()), dim3(THREADS), SMEM_BYTES, s, w0, w1, x0, x1,
                          p);
}

}  // namespace

cudaError_t launch_ffn_tc_small(const Cfg& c, const void* xperm, const int32_t* expert_start,
                          const int32_t* kept_counts, const void* w_gate_up, const void* w_down,
                          const void* x, const void* shared_gate_up, const void* shared_down,
                          void* yperm, void* yshared, void* h, int* status, cudaStream_t s) {
  const bool sh = c.Fs > 0;
  __nv_bfloat16* h_routed = static_cast<__nv_bfloat16*>(h);
  __nv_bfloat16* h_shared = h_routed + (size_t)c.send_rows * c.F;
  CUtensorMap w0, w1, x0, x1;
  // G1: weights [E*2F, d] / [2Fs, d] in 64-row boxes; tokens [A, d] / [N, d]
  if (!make_map(&w0, w_gate_up, c.d, (uint64_t)c.E * 2 * c.F, BW / 2) ||
      !make_map(&x0, xperm, c.d, c.send_rows, PIECE))
    return cudaErrorInvalidValue;
  w1 = w0;
  x1 = x0;
  if (sh && (!make_map(&w1, shared_gate_up, c.d, 2 * c.Fs, BW / 2) ||
             !make_map(&x1, x, c.d, c.N, PIECE)))
    return cudaErrorInvalidValue;
  TcParams p{expert_start, kept_counts, h_routed, h_shared, status,
             c.E, sh ? c.N : 0, c.d, c.F, c.Fs};
  cudaError_t e = launch<GATE_UP>(w0, w1, x0, x1, p, s);
  if (e != cudaSuccess) return e;
  // G2: weights [E*d, F] / [d, Fs] in 112-row boxes; tokens = h [A, F] / [N, Fs]
  if (!make_map(&w0, w_down, c.F, (uint64_t)c.E * c.d, BW2) ||
      !make_map(&x0, h_routed, c.F, c.send_rows, PIECE))
    return cudaErrorInvalidValue;
  w1 = w0;
  x1 = x0;
  if (sh && (!make_map(&w1, shared_down, c.Fs, c.d, BW2) ||
             !make_map(&x1, h_shared, c.Fs, c.N, PIECE)))
    return cudaErrorInvalidValue;
  p.out0 = static_cast<__nv_bfloat16*>(yperm);
  p.out1 = static_cast<__nv_bfloat16*>(yshared);
  return launch<DOWN>(w0, w1, x0, x1, p, s);
}

}  // namespace moe
