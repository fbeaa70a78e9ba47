// ffn_bwd_tc.cu -- backward of the grouped SwiGLU expert FFN on the tensor cores (bf16).
//
// Forward (Ultralytics glossary "Expert Parallelism", section "How tokens move
// between GPUs", step 3; fudan-mlsys-cn chapter 10, section 10.5 for the shared
// expert), per row x of an expert segment: g = Wg x, u = Wu x, h = silu(g) * u,
// y = Wd h.  Backward from dy (= w * dout for a routed row, dout for the shared one):
//   R1  gu, h  = recompute [g | u] = X W_gu^T with h = silu(g) * u    (M rows, N 2F, K d)
//   D1  dh = dY Wd, fused: dg = dh * u * silu'(g), du = dh * silu(g)  (M rows, N F,  K d)
//   D2  dX = [dg | du] W_gu                                           (M rows, N d,  K 2F)
//   W1  dWd[e]   = dY_e^T H_e                                          (M d,    N F,  K rows_e)
//   W2  dW_gu[e] = [dG | dU]_e^T X_e                                   (M 2F,   N d,  K rows_e)
// with silu'(z) = s(z) (1 + z (1 - s(z))), s = logistic.  g, u, h and [dg | du] are
// bf16 in a workspace; every product accumulates in fp32 in TMEM.
//
// One persistent kernel per kind, one CTA per SM, warp-specialised as the forward
// kernel: warp 0 TMA producer into a 4-stage ring (128-byte swizzle), warp 1 TMEM owner
// and single-thread tcgen05.mma issuer (M=128, N=256, K=16), warps 2-5 epilogue.
// Operands whose reduction index is not the contiguous one (W_down and W_gate_up in
// D1/D2, both operands of W1/W2) are loaded as MN-major tiles: 64-element x 64-row
// TMA boxes, one 128-byte row per K index, descriptors with a leading offset of one
// box (8 KiB) between 64-element MN chunks and 1 KiB between 8-row K groups, and the
// instruction descriptor's transpose bit for that operand.
// Every routed operand and result row is in the send-buffer layout (expert e's rows at
// expert_start[e]).  W1/W2 sum over a segment's rows, so the last K block of a segment
// must not add the next segment's rows (or send-buffer rows never written): in that
// block only the K=16 MMAs that reach the segment's rows are issued, and the rows past
// its end inside the last of them are zeroed by the MMA warp in both operands'
// shared-memory tiles (whole 128-byte rows, so the swizzle does not matter) before the
// MMA reads them.  The shared expert's rows end where its tensors end, and TMA fills the
// rest of a block with zeros.
// Experts with no rows get no W tiles; their gradients are written as zeros by the W
// kinds' epilogue warps, interleaved with the tiles (TMA stores of a zeroed box).
// The W kinds' K loops are short (one segment's rows), so their output write is the
// critical path: every epilogue warp stages its 32 rows of each 64-column box in shared
// memory (128-byte swizzle, two alternating 4 KB buffers per warp) and writes it with a
// TMA tensor store into [segments, M, N] maps that clip a segment's row tail, without
// waiting for the other warps; the ring has 3 stages there to make room.
// Every mbarrier wait is bounded (about 2 s) and reports through the status word.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
// W kinds: every epilogue warp stages its 32 rows of one 64-column box of the output
// tile (4 KB) for a TMA store, in two alternating buffers
constexpr int WBOX_BYTES = 32 * 64 * 2;
constexpr int OUT_BYTES = 4 * 2 * WBOX_BYTES;
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_BYTES = BN * BK * 2;   // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int BOX_BYTES = 64 * BK * 2;  // one MN-major box: 64 elements x 64 K rows
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;
constexpr int MAX_SEG = kMaxExperts + 1;
constexpr uint64_t WAIT_NS = 2000000000ull;

enum Kind { R1 = 0, D1 = 1, D2 = 2, W1 = 3, W2 = 4 };

template <int KIND>
struct Traits {
  static constexpr bool a_mn = KIND == W1 || KIND == W2;   // A loaded MN-major
  static constexpr bool b_mn = KIND != R1;                  // B loaded MN-major
  static constexpr bool k_rows = KIND == W1 || KIND == W2;  // reduction over segment rows
  // W kinds: short K loops (a segment's rows) make the output write the critical path;
  // the tile goes out through a 16 KB shared-memory box and TMA stores
  static constexpr bool tma_out = k_rows;
  static constexpr int stages = k_rows ? 3 : STAGES;  // room for the staging buffers
  static constexpr uint32_t idesc =
      idesc_bf16_f32(BM, BN) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16);
};

struct BwdParams {
  const int32_t* expert_start;
  const int32_t* kept_counts;
  __nv_bfloat16* out0;  // routed output   R1 gu, D1 dgu, D2 dx, W1 dWd, W2 dWgu
  __nv_bfloat16* out1;  // shared output
  __nv_bfloat16* aux0;  // R1: h out (routed) / D1: gu in (routed)
  __nv_bfloat16* aux1;  // shared counterpart
  int* err;
  int E, n_shared, d, F, Fs;
  int padded_layout;  // capacity-padded send buffer: rows between experts never written
};

struct Ctl {
  uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], drain;
  uint32_t tmem_base;
  int abort;
  int kept_end;  // end of the routed rows written in the send buffer (packed layout)
  int n_empty;   // W kinds: routed experts with no rows, whose gradient is written as zeros
  int empty_ids[kMaxExperts];
  int tile_start[MAX_SEG + 1];
  int mtiles[MAX_SEG];
  int rows[MAX_SEG];
  int row_base[MAX_SEG];  // first row of the segment in the send buffer (0: shared)
};

template <int KIND>
constexpr size_t smem_bytes() {
  return 1024 + (size_t)Traits<KIND>::stages * STAGE_BYTES +
         (Traits<KIND>::tma_out ? OUT_BYTES + WBOX_BYTES : 0) + sizeof(Ctl);
}

// TMA store of one 64-column x 32-row box of a [segments, M, N] tensor (rows past a
// segment's M are clipped by the map); the caller commits it to its bulk group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x,
                                             int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(z), "r"(saddr(src))
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// the shared-memory sources of this thread's bulk stores, all but the latest group,
// have been read
__device__ __forceinline__ void bulk_wait_read_prev() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// this thread's bulk stores have completed
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}


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

// MN-major 128-byte-swizzle descriptor: start >> 4, leading offset = one 64-element
// box (between MN chunks), stride offset 1 KiB (between 8-row K groups).
__device__ __forceinline__ uint64_t sdesc_mn(uint32_t a) {
  return (uint64_t)((a & 0x3FFFFu) >> 4) | ((uint64_t)(BOX_BYTES >> 4) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// ---------------------------------------------------------------- geometry
// Output extents of a segment: M (rows of the result), N (columns), K (reduction).
template <int KIND>
__device__ __forceinline__ void extents(bool routed, int rows, const BwdParams& p, int* M, int* N,
                                        int* K) {
  const int Fx = routed ? p.F : p.Fs;
  switch (KIND) {
    case R1: *M = rows; *N = Fx; *K = p.d; break;       // N counts hidden units (g and u)
    case D1: *M = rows; *N = Fx; *K = p.d; break;
    case D2: *M = rows; *N = p.d; *K = 2 * Fx; break;
    case W1: *M = p.d; *N = Fx; *K = rows; break;
    default: *M = 2 * Fx; *N = p.d; *K = rows; break;   // W2
  }
}

template <int KIND>
__device__ __forceinline__ int n_step() { return KIND == R1 ? BN / 2 : BN; }

struct Tile {
  int seg, m0, n0, M, N, K, row_base;
  bool routed;
};

template <int KIND>
__device__ __forceinline__ Tile decode(const Ctl* ctl, int nseg, int t, const BwdParams& p) {
  int lo = 0, hi = nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ctl->tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  Tile tl;
  tl.seg = lo;
  tl.routed = lo < p.E;
  extents<KIND>(tl.routed, ctl->rows[lo], p, &tl.M, &tl.N, &tl.K);
  const int local = t - ctl->tile_start[lo];
  if (Traits<KIND>::k_rows) {
    // W kinds: column tiles fastest, so that the CTAs running at the same time write
    // whole contiguous rows of dW (the write stream is the bound there)
    const int nt = (tl.N + n_step<KIND>() - 1) / n_step<KIND>();
    tl.m0 = (local / nt) * BM;
    tl.n0 = (local % nt) * n_step<KIND>();
  } else {
    // column-tile major: CTAs running at the same time share a weight tile in L2
    const int mt = ctl->mtiles[lo];
    tl.m0 = (local % mt) * BM;
    tl.n0 = (local / mt) * n_step<KIND>();
  }
  tl.row_base = ctl->row_base[lo];
  return tl;
}

// ---------------------------------------------------------------- kernel
template <int KIND>
__global__ void __launch_bounds__(THREADS, 1)
ffn_bwd_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
               const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
               const __grid_constant__ CUtensorMap tmO0, const __grid_constant__ CUtensorMap tmO1,
               BwdParams p) {
  using Tr = Traits<KIND>;
  constexpr int NST = Tr::stages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stage_out = smem + (size_t)NST * STAGE_BYTES;  // W kinds only
  uint8_t* zero_box = stage_out + OUT_BYTES;               // W kinds: 4 KB of zeros
  Ctl* ctl = reinterpret_cast<Ctl*>(stage_out + (Tr::tma_out ? OUT_BYTES + WBOX_BYTES : 0));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nseg = p.E + (p.n_shared > 0 ? 1 : 0);

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < NST; ++s) {
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
  }
  if (warp == 1) tmem_alloc(&ctl->tmem_base, TMEM_COLS);
  if (warp == 2) {  // per-segment tile table
    int base = 0;
    for (int s0 = 0; s0 < nseg; s0 += 32) {
      const int s = s0 + lane;
      int v = 0;
      if (s < nseg) {
        const bool routed = s < p.E;
        const int cnt = routed ? p.kept_counts[s] : p.n_shared;
        int M, N, K;
        extents<KIND>(routed, cnt, p, &M, &N, &K);
        const int mt = (M + BM - 1) / BM;
        ctl->mtiles[s] = mt > 0 ? mt : 1;
        ctl->rows[s] = cnt;
        ctl->row_base[s] = routed ? p.expert_start[s] : 0;
        // a segment with no rows has nothing to compute (W kinds: its gradient is zeroed
        // elsewhere)
        v = (cnt > 0) ? mt * ((N + n_step<KIND>() - 1) / n_step<KIND>()) : 0;
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
    if (lane == 0) {
      ctl->tile_start[nseg] = base;
      int end = 0;
      for (int s = 0; s < p.E; ++s)
        if (ctl->rows[s] > 0 && ctl->row_base[s] + ctl->rows[s] > end)
          end = ctl->row_base[s] + ctl->rows[s];
      ctl->kept_end = end;
      int ne = 0;
      if (Tr::k_rows)
        for (int s = 0; s < p.E; ++s)
          if (ctl->rows[s] == 0) ctl->empty_ids[ne++] = s;
      ctl->n_empty = ne;
    }
  }
  if (Tr::tma_out) {
    for (int i = threadIdx.x; i < WBOX_BYTES / 16; i += blockDim.x)
      reinterpret_cast<uint4*>(zero_box)[i] = make_uint4(0, 0, 0, 0);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile tl = decode<KIND>(ctl, nseg, t, p);
        const CUtensorMap* ma = tl.routed ? &tmA0 : &tmA1;
        const CUtensorMap* mb = tl.routed ? &tmB0 : &tmB1;
        const int Fx = tl.routed ? p.F : p.Fs;
        for (int k0 = 0; k0 < tl.K; k0 += BK) {
          if (!mbar_wait(&ctl->empty[stage], phase ^ 1, ctl, p.err, 1)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + (size_t)stage * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          mbar_expect_tx(&ctl->full[stage], STAGE_BYTES);
          uint64_t* fb = &ctl->full[stage];
          if (KIND == R1) {
            // A rows of the segment (K-major); B = 128 gate rows and the matching up rows
            const int wrow = (tl.routed ? tl.seg * 2 * p.F : 0) + tl.n0;
            tma_load(sa, ma, fb, k0, tl.row_base + tl.m0);
            tma_load(sb, mb, fb, k0, wrow);
            tma_load(sb + B_BYTES / 2, mb, fb, k0, wrow + Fx);
          } else if (KIND == D1 || KIND == D2) {
            // A rows (K-major); B MN-major boxes of the weight [K rows, N columns]
            const int wk = (tl.routed ? tl.seg * (KIND == D1 ? p.d : 2 * p.F) : 0) + k0;
            tma_load(sa, ma, fb, k0, tl.row_base + tl.m0);
#pragma unroll
            for (int j = 0; j < 4; ++j) tma_load(sb + j * BOX_BYTES, mb, fb, tl.n0 + 64 * j, wk);
          } else {
            // W1/W2: both operands MN-major over the segment's rows
            const int r0 = tl.row_base + k0;
#pragma unroll
            for (int j = 0; j < 2; ++j) tma_load(sa + j * BOX_BYTES, ma, fb, tl.m0 + 64 * j, r0);
#pragma unroll
            for (int j = 0; j < 4; ++j) tma_load(sb + j * BOX_BYTES, mb, fb, tl.n0 + 64 * j, r0);
          }
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == NST) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {  // let this CTA's copies land before the CTA goes away
        const uint64_t t0 = now_ns();
        for (int s = 0; s < NST; ++s)
          if (armed >> s & 1u)
            while (!mbar_try_wait(&ctl->full[s], armed_parity >> s & 1u) &&
                   now_ns() - t0 < WAIT_NS) {
            }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (whole warp: the K-tail
    // zeroing of W kinds is shared by its lanes; lane 0 issues)
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true, issued = false;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = decode<KIND>(ctl, nseg, t, p);
      bool got = true;
      if (lane == 0) got = mbar_wait(&ctl->tempty[acc], acc_phase ^ 1, ctl, p.err, 2);
      if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t dt = tmem_base + (uint32_t)(acc * BN);
      for (int k0 = 0; k0 < tl.K; k0 += BK) {
        if (lane == 0) got = mbar_wait(&ctl->full[stage], phase, ctl, p.err, 3);
        if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem + (size_t)stage * STAGE_BYTES;
        int kk_end = BK / 16;  // MMAs (K = 16 each) of this block
        if (Tr::k_rows && tl.routed && k0 + BK > tl.K) {
          // the segment ends inside this block: only the MMAs that reach its rows run,
          // and the rows past its end inside the last of them (rows rem .. 16*kk_end-1)
          // are zeroed by the whole warp, whole 128-byte rows at a time, before the MMA
          // reads them: in A's 2 boxes always (B's rows there are the following
          // segments', finite values, so their products vanish), in B's 4 boxes too
          // where those rows may never have been written (past the last written row of
          // the packed layout, or anywhere in the padded one)
          const int rem = tl.K - k0;
          kk_end = (rem + 15) >> 4;
          const int zr1 = kk_end * 16;
          if (rem < zr1) {
            const uint4 z = make_uint4(0, 0, 0, 0);
            const bool b_unwritten =
                p.padded_layout || tl.row_base + k0 + zr1 > ctl->kept_end;
            const int nbox = b_unwritten ? 6 : 2;
            for (int box = 0; box < nbox; ++box) {
              uint8_t* base = box < 2 ? sa + box * BOX_BYTES : sa + A_BYTES + (box - 2) * BOX_BYTES;
              for (int row = rem + (lane >> 3); row < zr1; row += 4)
                *reinterpret_cast<uint4*>(base + row * 128 + (lane & 7) * 16) = z;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          }
          __syncwarp();
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t a0 = saddr(sa);
          const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if (kk >= kk_end) break;
            const uint64_t ad = Tr::a_mn ? sdesc_mn(a0 + kk * 2048) : sdesc(a0 + kk * 32);
            const uint64_t bd = Tr::b_mn ? sdesc_mn(b0 + kk * 2048) : sdesc(b0 + kk * 32);
            tc_mma(dt, ad, bd, Tr::idesc, (k0 > 0 || kk > 0) ? 1u : 0u);
          }
          issued = true;
          tc_commit(&ctl->empty[stage]);
        }
        __syncwarp();
        if (++stage == NST) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(&ctl->tfull[acc]);
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (lane == 0 && issued) {  // every MMA of this thread has finished before TMEM is freed
      tc_commit(&ctl->drain);
      const uint64_t t0 = now_ns();
      while (!mbar_try_wait(&ctl->drain, 0) && now_ns() - t0 < WAIT_NS) {
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue (warps 2-5)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    // W kinds: the gradients of experts with no rows are zeros, written here as 32-row x
    // 64-column TMA stores of a zeroed box; the boxes are spread over every epilogue warp
    // of the grid and issued a few after each tile, while the MMAs of the next run
    int zn = 0, znbn = 1, zpe = 1, zper = 0, z = 0, zstride = 0;
    if (Tr::tma_out) {
      int M, N, K;
      extents<KIND>(true, 1, p, &M, &N, &K);
      znbn = (N + 63) / 64;             // boxes across a row of dW
      zpe = ((M + 31) / 32) * znbn;     // boxes per expert
      zn = ctl->n_empty * zpe;
      z = blockIdx.x * 4 + q;
      zstride = gridDim.x * 4;
      const int mine = z < zn ? (zn - z + zstride - 1) / zstride : 0;
      const int tiles = blockIdx.x < total ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
      zper = tiles > 0 ? (mine + tiles - 1) / tiles : mine;
    }
    auto zero_boxes = [&](int count) {
      for (int i = 0; i < count && z < zn; ++i, z += zstride) {
        if (lane == 0) {
          const int e = ctl->empty_ids[z / zpe], b = z % zpe;
          tma_store_3d(&tmO0, zero_box, (b % znbn) * 64, (b / znbn) * 32, e);
          bulk_commit();
        }
      }
    };
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = decode<KIND>(ctl, nseg, t, p);
      const int Fx = tl.routed ? p.F : p.Fs;
      if (!mbar_wait(&ctl->tfull[acc], acc_phase, ctl, p.err, 4)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      const bool valid = tl.m0 + r < tl.M;
      __nv_bfloat16* out = tl.routed ? p.out0 : p.out1;
      if (KIND == R1) {
        // g in columns [0,128), u in [128,256): gu row (g at f, u at Fx + f) and h
        const int64_t row = tl.row_base + tl.m0 + r;
        __nv_bfloat16* gurow = out + row * (2 * Fx);
        __nv_bfloat16* hrow = (tl.routed ? p.aux0 : p.aux1) + row * Fx;
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(tb + c, g);
          tmem_ld32(tb + BN / 2 + c, u);
          tmem_ld_wait(g);
          tmem_ld_wait(u);
          if (valid) {
            uint32_t pg[16], pu[16], ph[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
              const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
              pg[i] = pack_bf16(g0, g1);
              pu[i] = pack_bf16(u0, u1);
              // the forward's expression, so that recomputed h equals the saved one
              ph[i] = pack_bf16(__fdividef(g0, 1.0f + __expf(-g0)) * u0,
                                __fdividef(g1, 1.0f + __expf(-g1)) * u1);
            }
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int col = tl.n0 + c + v * 8;
              if (col < Fx) {
                *reinterpret_cast<uint4*>(gurow + col) =
                    make_uint4(pg[4 * v], pg[4 * v + 1], pg[4 * v + 2], pg[4 * v + 3]);
                *reinterpret_cast<uint4*>(gurow + Fx + col) =
                    make_uint4(pu[4 * v], pu[4 * v + 1], pu[4 * v + 2], pu[4 * v + 3]);
                *reinterpret_cast<uint4*>(hrow + col) =
                    make_uint4(ph[4 * v], ph[4 * v + 1], ph[4 * v + 2], ph[4 * v + 3]);
              }
            }
          }
        }
      } else if (KIND == D1) {
        // dh columns [n0, n0+256): dg = dh u silu'(g), du = dh silu(g), from gu
        const int64_t row = tl.row_base + tl.m0 + r;
        const __nv_bfloat16* gurow = (tl.routed ? p.aux0 : p.aux1) + row * (2 * Fx);
        __nv_bfloat16* drow = out + row * (2 * Fx);
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t dh[32];
          tmem_ld32(tb + c, dh);
          tmem_ld_wait(dh);
          if (valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int col = tl.n0 + c + v * 8;
              if (col >= Fx) continue;
              const uint4 gv = *reinterpret_cast<const uint4*>(gurow + col);
              const uint4 uv = *reinterpret_cast<const uint4*>(gurow + Fx + col);
              const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
              const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
              uint32_t pdg[4], pdu[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                float dgo[2], duo[2];
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                  const float g = __uint_as_float(h2 ? (gw[i] & 0xffff0000u) : (gw[i] << 16));
                  const float u = __uint_as_float(h2 ? (uw[i] & 0xffff0000u) : (uw[i] << 16));
                  const float d = __uint_as_float(dh[v * 8 + 2 * i + h2]);
                  const float s = 1.0f / (1.0f + __expf(-g));
                  dgo[h2] = d * u * s * (1.0f + g * (1.0f - s));
                  duo[h2] = d * g * s;
                }
                pdg[i] = pack_bf16(dgo[0], dgo[1]);
                pdu[i] = pack_bf16(duo[0], duo[1]);
              }
              *reinterpret_cast<uint4*>(drow + col) = make_uint4(pdg[0], pdg[1], pdg[2], pdg[3]);
              *reinterpret_cast<uint4*>(drow + Fx + col) =
                  make_uint4(pdu[0], pdu[1], pdu[2], pdu[3]);
            }
          }
        }
      } else if (Tr::tma_out) {
        // [M, N] tile of dW, one 64-column box at a time: each warp moves its 32 rows
        // TMEM -> registers -> its own 4 KB staging buffer (128-byte swizzle: 16-byte
        // chunk j of row r at r*128 + (j^(r&7))*16) -> one TMA store, alternating two
        // buffers so that staging a box overlaps the previous box's store; no warp waits
        // for another.  Every box commits one bulk group (empty when the box lies past
        // the last column), so waiting until all but the latest group have read their
        // source frees the buffer about to be written.
        uint8_t* wst = stage_out + (size_t)q * 2 * WBOX_BYTES;
#pragma unroll 1
        for (int bx = 0; bx < BN / 64; ++bx) {
          uint32_t y[2][32];
          tmem_ld32(tb + 64 * bx, y[0]);
          tmem_ld32(tb + 64 * bx + 32, y[1]);
          tmem_ld_wait(y[0]);
          tmem_regs_ready(y[1]);
          if (bx == BN / 64 - 1) {  // the accumulator goes back to the MMA warp
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->tempty[acc]);
          }
          uint8_t* buf = wst + (size_t)(bx & 1) * WBOX_BYTES;
          if (lane == 0) bulk_wait_read_prev();
          __syncwarp();
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16(__uint_as_float(y[h2][2 * i]), __uint_as_float(y[h2][2 * i + 1]));
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int chunk = h2 * 4 + v;
              *reinterpret_cast<uint4*>(buf + lane * 128 + ((chunk ^ (lane & 7)) << 4)) =
                  make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            if (tl.n0 + 64 * bx < tl.N)
              tma_store_3d(tl.routed ? &tmO0 : &tmO1, buf, tl.n0 + 64 * bx, tl.m0 + q * 32,
                           tl.routed ? tl.seg : 0);
            bulk_commit();
          }
        }
        zero_boxes(zper);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
        continue;
      } else {
        // plain bf16 store of the [M, N] result
        __nv_bfloat16* orow;
        if (KIND == D2) {
          orow = out + (int64_t)(tl.row_base + tl.m0 + r) * tl.N;
        } else {
          const int64_t seg_off = tl.routed ? (int64_t)tl.seg * tl.M * tl.N : 0;
          orow = out + seg_off + (int64_t)(tl.m0 + r) * tl.N;
        }
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
              if (col < tl.N)
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
    if (Tr::tma_out) {
      zero_boxes(zn);  // what is left (all of it in a CTA without tiles)
      if (lane == 0) bulk_wait_all();
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

// 2-D bf16 map over a row-major [rows, cols] matrix; box = box_cols x box_rows.
// K-major tiles: box 64 columns (the reduction index) x 128 / 256 rows.
// MN-major tiles: box 64 columns (output index) x 64 rows (the reduction index).
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
              uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 map over [segs, rows, cols] (row-major), box 64 columns x 128 rows x 1,
// 128-byte swizzle: the destination of the W kinds' tile stores.
bool make_out_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                  uint64_t segs) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {cols, rows, segs};
  const cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
  const cuuint32_t box[3] = {64, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KIND>
cudaError_t run(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
                const CUtensorMap& b1, const CUtensorMap& o0, const CUtensorMap& o1,
                const BwdParams& p, cudaStream_t s) {
  auto k = ffn_bwd_kernel<KIND>;
  constexpr size_t bytes = smem_bytes<KIND>();
  static_assert(bytes <= 232448, "shared memory per CTA");
  static bool attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_set[dev & 63]) {
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    attr_set[dev & 63] = true;
  }
  k<<<num_sms(), THREADS, bytes, s>>>(a0, a1, b0, b1, o0, o1, p);
  return cudaGetLastError();
}

}  // namespace

size_t saved_bytes(const Cfg& c) {
  return 2 * 3 * ((size_t)c.send_rows * c.F + (size_t)c.N * c.Fs);
}

size_t ffn_backward_ws_bytes(const Cfg& c) {
  // bf16, send-buffer layout: gu [S, 2F] + [N, 2Fs]; h [S, F] + [N, Fs]; dgu [S, 2F] +
  // [N, 2Fs]
  const size_t S = (size_t)c.send_rows, n = (size_t)c.N;
  return 2 * (S * 5 * (size_t)c.F + n * 5 * (size_t)c.Fs);
}

cudaError_t launch_ffn_backward(const Cfg& c, const void* xperm, const int32_t* expert_start,
                                const int32_t* kept_counts, const void* w_gate_up,
                                const void* w_down, const void* x, const void* shared_gate_up,
                                const void* shared_down, const void* dyperm, const void* dout,
                                void* dxperm, void* dx_shared, void* dw_gate_up, void* dw_down,
                                void* dshared_gate_up, void* dshared_down, const void* saved,
                                void* ws, int* status, cudaStream_t s) {
  using bf = __nv_bfloat16;
  const bool sh = c.Fs > 0;
  const uint64_t N = (uint64_t)c.N, d = (uint64_t)c.d;
  const uint64_t F = (uint64_t)c.F, Fs = (uint64_t)c.Fs, E = (uint64_t)c.E;
  const uint64_t S = (uint64_t)c.send_rows;  // rows of the send buffer
  bf* gu = static_cast<bf*>(ws);
  bf* gu_s = gu + S * 2 * F;
  bf* h = gu_s + N * 2 * Fs;
  bf* h_s = h + S * F;
  bf* dgu = h_s + N * Fs;
  bf* dgu_s = dgu + S * 2 * F;
  cudaError_t e;
  BwdParams p{expert_start, kept_counts, nullptr, nullptr, nullptr, nullptr, status,
              c.E, sh ? c.N : 0, c.d, c.F, c.Fs, c.mode == MOE_DISPATCH_CAPACITY_PADDED ? 1 : 0};
  CUtensorMap a0, a1, b0, b1, o0, o1;
  // activations kept by the forward (moe_expert_ffn_save), in the send-buffer layout:
  // h [S, F] + [N, Fs], then g|u [S, 2F] + [N, 2Fs]; otherwise R1 recomputes them
  const bf* sv_h = static_cast<const bf*>(saved);
  const bf* sv_hs = sv_h ? sv_h + S * F : nullptr;
  const bf* sv_gu = sv_h ? sv_hs + N * Fs : nullptr;
  const bf* sv_gus = sv_h ? sv_gu + S * 2 * F : nullptr;
  const bf* hr = saved ? sv_h : h;      // h as W1 reads it
  const bf* hrs = saved ? sv_hs : h_s;
  // R1: A = xperm / x (K-major over d); B = W_gu rows (K-major)
  if (!make_map(&a0, xperm, d, S, 64, BM) || !make_map(&b0, w_gate_up, d, E * 2 * F, 64, BN / 2))
    return cudaErrorInvalidValue;
  a1 = a0;
  b1 = b0;
  if (sh && (!make_map(&a1, x, d, N, 64, BM) || !make_map(&b1, shared_gate_up, d, 2 * Fs, 64, BN / 2)))
    return cudaErrorInvalidValue;
  p.out0 = gu; p.out1 = gu_s; p.aux0 = h; p.aux1 = h_s;
  if (!saved && (e = run<R1>(a0, a1, b0, b1, a0, a0, p, s)) != cudaSuccess) return e;
  // D1: A = dY (K-major over d); B = W_down as [d rows, F columns], MN-major
  if (!make_map(&a0, dyperm, d, S, 64, BM) || !make_map(&b0, w_down, F, E * d, 64, 64))
    return cudaErrorInvalidValue;
  a1 = a0;
  b1 = b0;
  if (sh && (!make_map(&a1, dout, d, N, 64, BM) || !make_map(&b1, shared_down, Fs, d, 64, 64)))
    return cudaErrorInvalidValue;
  p.out0 = dgu; p.out1 = dgu_s;
  p.aux0 = saved ? const_cast<bf*>(sv_gu) : gu;
  p.aux1 = saved ? const_cast<bf*>(sv_gus) : gu_s;
  if ((e = run<D1>(a0, a1, b0, b1, a0, a0, p, s)) != cudaSuccess) return e;
  // D2: A = [dG | dU] (K-major over 2F); B = W_gu as [2F rows, d columns], MN-major
  if (!make_map(&a0, dgu, 2 * F, S, 64, BM) || !make_map(&b0, w_gate_up, d, E * 2 * F, 64, 64))
    return cudaErrorInvalidValue;
  a1 = a0;
  b1 = b0;
  if (sh && (!make_map(&a1, dgu_s, 2 * Fs, N, 64, BM) || !make_map(&b1, shared_gate_up, d, 2 * Fs, 64, 64)))
    return cudaErrorInvalidValue;
  p.out0 = static_cast<bf*>(dxperm); p.out1 = static_cast<bf*>(dx_shared);
  p.aux0 = p.aux1 = nullptr;
  if ((e = run<D2>(a0, a1, b0, b1, a0, a0, p, s)) != cudaSuccess) return e;
  // W1: dWd[e] = dY_e^T H_e: A = dY MN-major ([rows, d]), B = H MN-major ([rows, F])
  if (!make_map(&a0, dyperm, d, S, 64, 64) || !make_map(&b0, hr, F, S, 64, 64))
    return cudaErrorInvalidValue;
  a1 = a0;
  b1 = b0;
  if (sh && (!make_map(&a1, dout, d, N, 64, 64) ||
             !make_map(&b1, hrs, Fs, N, 64, 64)))
    return cudaErrorInvalidValue;
  // dWd [E, d, F] and the shared [d, Fs], written by TMA stores
  if (!make_out_map(&o0, dw_down, F, d, E)) return cudaErrorInvalidValue;
  o1 = o0;
  if (sh && !make_out_map(&o1, dshared_down, Fs, d, 1)) return cudaErrorInvalidValue;
  p.out0 = static_cast<bf*>(dw_down); p.out1 = static_cast<bf*>(dshared_down);
  if ((e = run<W1>(a0, a1, b0, b1, o0, o1, p, s)) != cudaSuccess) return e;
  // W2: dW_gu[e] = [dG | dU]_e^T X_e: A = dGU MN-major ([rows, 2F]), B = X MN-major
  if (!make_map(&a0, dgu, 2 * F, S, 64, 64) || !make_map(&b0, xperm, d, S, 64, 64))
    return cudaErrorInvalidValue;
  a1 = a0;
  b1 = b0;
  if (sh && (!make_map(&a1, dgu_s, 2 * Fs, N, 64, 64) || !make_map(&b1, x, d, N, 64, 64)))
    return cudaErrorInvalidValue;
  // dW_gu [E, 2F, d] and the shared [2Fs, d]
  if (!make_out_map(&o0, dw_gate_up, d, 2 * F, E)) return cudaErrorInvalidValue;
  o1 = o0;
  if (sh && !make_out_map(&o1, dshared_gate_up, d, 2 * Fs, 1)) return cudaErrorInvalidValue;
  p.out0 = static_cast<bf*>(dw_gate_up); p.out1 = static_cast<bf*>(dshared_gate_up);
  return run<W2>(a0, a1, b0, b1, o0, o1, p, s);
}

}  // namespace moe
