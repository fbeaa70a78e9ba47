// dispatch.cu -- counting, capacity, send-order slots, and the permute (dispatch).
//
// Ultralytics glossary "Expert Parallelism", section "How tokens move between GPUs",
// step 2 and its example: count token-expert assignments per expert and per device,
// and send each token's hidden state to the device holding its expert.  Section
// "Load balancing and capacity": an expert accepts at most a fixed number of
// tokens per batch (cf times its even share); the overflow skips that expert.
//
// Single-GPU form: the "send buffer" xperm holds the kept rows in the order an
// all-to-all would send them (rank, then expert, then token order), and the
// per-rank counts/offsets are its split sizes.  Deterministic, no inter-CTA waits:
//   K2a count   one CTA per chunk of kChunk assignments (in priority order): per-chunk
//               histogram; the capacity-padded layout also clears perm_src here
//   K2b scan    one CTA: per-expert prefix over chunks (chunk bases), routed counts,
//               kept = min(count, C), send-order expert starts, rank counts/offsets
//   K2c assign  one CTA per chunk: stable (token-order) rank of each assignment
//               within its expert -> slot or drop; perm_src tail cleared
//   K3  permute every token row read once, written to each of its kept slots
//               (16-byte vector loads / stores)

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int T2 = 256;  // threads of the count / scan / assign kernels

// Assignments compete for capacity in priority order p = 0..A-1.  Packed: p is the
// assignment index a = t*k + j (token order).  Capacity-padded: p = j*N + t, every
// token's first choice before any second choice (choice-major).
__device__ __forceinline__ int64_t assignment_of(int64_t p, int N, int k, int mode) {
  return mode == MOE_DISPATCH_CAPACITY_PADDED ? (p % N) * k + p / N : p;
}

// The three passes are device functions of a chunk index `blk` (of `nblk`), run as one
// kernel each, or back to back by one CTA when the assignments fit in one chunk.
__device__ __forceinline__ void count_pass(int blk, int nblk, const int32_t* __restrict__ idx,
                                           int64_t A, int N, int k, int E, int mode,
                                           int32_t* __restrict__ chunk_hist,
                                           int32_t* __restrict__ perm_src, int64_t send_rows) {
  __shared__ int hist[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += T2) hist[e] = 0;
  __syncthreads();
  const int64_t p0 = (int64_t)blk * kChunk;
  const int64_t p1 = min(p0 + kChunk, A);
  for (int64_t p = p0 + threadIdx.x; p < p1; p += T2) {
    const int e = idx[assignment_of(p, N, k, mode)];
    if ((unsigned)e < (unsigned)E) atomicAdd(&hist[e], 1);
  }
  // padded layout: rows without an assignment hold -1 (the assign kernel, which runs
  // after this one, overwrites the kept rows)
  if (mode == MOE_DISPATCH_CAPACITY_PADDED)
    for (int64_t r = (int64_t)blk * T2 + threadIdx.x; r < send_rows; r += (int64_t)nblk * T2)
      perm_src[r] = -1;
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += T2) chunk_hist[(int64_t)blk * E + e] = hist[e];
}

__global__ void __launch_bounds__(T2)
count_kernel(const int32_t* __restrict__ idx, int64_t A, int N, int k, int E, int mode,
             int32_t* __restrict__ chunk_hist, int32_t* __restrict__ perm_src, int64_t send_rows) {
  count_pass(blockIdx.x, gridDim.x, idx, A, N, k, E, mode, chunk_hist, perm_src, send_rows);
}

// Position of expert e in the send order (rank ascending, expert ascending).
__device__ __forceinline__ int send_pos(int e, int E, int R, int rank_map) {
  if (rank_map == MOE_RANK_ROUND_ROBIN) {
    const int r = e % R, j = e / R;
    const int q = E / R, rem = E % R;
    return r * q + min(r, rem) + j;  // ranks below r hold q (+1 for the first rem) experts
  }
  return e;
}

__device__ __forceinline__ void scan_pass(int32_t* __restrict__ chunk_hist, int n_chunks, int E,
                                          int R, int rank_map, int C, int mode,
                                          int32_t* __restrict__ expert_counts,
                                          int32_t* __restrict__ kept_counts,
                                          int32_t* __restrict__ expert_start,
                                          int32_t* __restrict__ rank_counts,
                                          int32_t* __restrict__ rank_offsets,
                                          int32_t* __restrict__ num_kept) {
  __shared__ int kept_by_pos[kMaxExperts];
  __shared__ int start_by_pos[kMaxExperts + 1];
  __shared__ int warp_tot[T2 / 32];
  const int e = threadIdx.x;
  int pos = 0, kept = 0;
  if (e < E) {
    int run = 0;
    for (int c = 0; c < n_chunks; ++c) {  // coalesced across e
      const int v = chunk_hist[(int64_t)c * E + e];
      chunk_hist[(int64_t)c * E + e] = run;  // becomes the chunk's base for expert e
      run += v;
    }
    kept = min(run, C);
    expert_counts[e] = run;
    kept_counts[e] = kept;
    pos = send_pos(e, E, R, rank_map);
    kept_by_pos[pos] = kept;
  }
  __syncthreads();
  // exclusive scan of kept_by_pos over E <= 256 positions (thread i = position i)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int v = (threadIdx.x < E) ? kept_by_pos[threadIdx.x] : 0;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += warp_tot[w];
  if (threadIdx.x < E) start_by_pos[threadIdx.x] = base + incl - v;
  if (threadIdx.x == E - 1) start_by_pos[E] = base + incl;
  __syncthreads();
  const bool padded = mode == MOE_DISPATCH_CAPACITY_PADDED;  // expert rows start at pos * C
  if (e < E) expert_start[e] = padded ? pos * C : start_by_pos[pos];
  // ranks: send positions of rank r are [P_r, P_{r+1})
  for (int r = threadIdx.x; r < R; r += T2) {
    int p0, p1;
    if (rank_map == MOE_RANK_ROUND_ROBIN) {
      const int q = E / R, rem = E % R;
      p0 = r * q + min(r, rem);
      p1 = p0 + q + (r < rem ? 1 : 0);
    } else {
      p0 = r * (E / R);
      p1 = p0 + E / R;
    }
    rank_offsets[r] = padded ? p0 * C : start_by_pos[p0];
    rank_counts[r] = start_by_pos[p1] - start_by_pos[p0];
    if (r == R - 1) rank_offsets[R] = padded ? p1 * C : start_by_pos[p1];
  }
  if (threadIdx.x == 0) *num_kept = start_by_pos[E];
}

__global__ void __launch_bounds__(T2)
scan_kernel(int32_t* __restrict__ chunk_hist, int n_chunks, int E, int R, int rank_map, int C,
            int mode,
            int32_t* __restrict__ expert_counts, int32_t* __restrict__ kept_counts,
            int32_t* __restrict__ expert_start, int32_t* __restrict__ rank_counts,
            int32_t* __restrict__ rank_offsets, int32_t* __restrict__ num_kept) {
  scan_pass(chunk_hist, n_chunks, E, R, rank_map, C, mode, expert_counts, kept_counts,
            expert_start, rank_counts, rank_offsets, num_kept);
}

__device__ __forceinline__ void assign_pass(int blk, const int32_t* __restrict__ idx, int64_t A,
                                            int N, int k, int E, int C, int mode,
                                            const int32_t* __restrict__ chunk_base,
                                            const int32_t* __restrict__ expert_start,
                                            const int32_t* __restrict__ num_kept,
                                            int32_t* __restrict__ slot_of,
                                            int32_t* __restrict__ perm_src) {
  __shared__ int run[kMaxExperts];
  __shared__ int wcnt[T2 / 32][kMaxExperts];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t a0 = (int64_t)blk * kChunk;
  const int64_t a1 = min(a0 + kChunk, A);
  for (int e = tid; e < E; e += T2) run[e] = chunk_base[(int64_t)blk * E + e];
  for (int64_t a = a0; a < a1; a += T2) {
    for (int q = tid; q < (T2 / 32) * E; q += T2) wcnt[q / E][q % E] = 0;
    __syncthreads();  // also orders run[] updates of the previous round
    const int64_t my = a + tid;  // priority index of this thread's assignment
    const int64_t asg = assignment_of(my, N, k, mode);
    int e = -1;
    if (my < a1) {
      e = idx[asg];
      if ((unsigned)e >= (unsigned)E) e = -1;
    }
    const int key = (e >= 0) ? e : -1 - lane;  // invalid lanes never group together
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    const int rank_in_warp = __popc(peers & lanemask_lt());
    if (e >= 0 && rank_in_warp == 0) wcnt[warp][e] = __popc(peers);
    __syncthreads();
    int pos = 0;
    if (e >= 0) {
      pos = run[e] + rank_in_warp;
      for (int w = 0; w < warp; ++w) pos += wcnt[w][e];
    }
    __syncthreads();
    for (int q = tid; q < E; q += T2) {
      int s = 0;
      for (int w = 0; w < T2 / 32; ++w) s += wcnt[w][q];
      run[q] += s;
    }
    if (my < a1) {
      if (e >= 0 && pos < C) {
        const int slot = expert_start[e] + pos;
        slot_of[asg] = slot;
        perm_src[slot] = (int32_t)asg;
      } else {
        slot_of[asg] = -1;
      }
    }
    __syncthreads();  // wcnt is cleared at the top of the next round
  }
  // packed layout: rows past num_kept carry no assignment
  if (mode == MOE_DISPATCH_PACKED) {
    const int nk = *num_kept;
    for (int64_t s = a0 + tid; s < a1; s += T2)
      if (s >= nk) perm_src[s] = -1;
  }
}

__global__ void __launch_bounds__(T2)
assign_kernel(const int32_t* __restrict__ idx, int64_t A, int N, int k, int E, int C, int mode,
              const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ expert_start,
              const int32_t* __restrict__ num_kept, int32_t* __restrict__ slot_of,
              int32_t* __restrict__ perm_src) {
  pdl_trigger();  // the permute kernel may be scheduled now; it waits for this one
  assign_pass(blockIdx.x, idx, A, N, k, E, C, mode, chunk_base, expert_start, num_kept, slot_of,
              perm_src);
}

// All of count, scan and assign for assignments that fit in one chunk (decode-sized
// batches): one CTA, the passes separated by block barriers (a pass's global writes
// are visible to the whole block after the barrier), one launch instead of three.
__global__ void __launch_bounds__(T2)
count_scan_assign_kernel(const int32_t* __restrict__ idx, int64_t A, int N, int k, int E, int R,
                         int rank_map, int C, int mode, int32_t* __restrict__ chunk_hist,
                         int32_t* __restrict__ expert_counts, int32_t* __restrict__ kept_counts,
                         int32_t* __restrict__ expert_start, int32_t* __restrict__ rank_counts,
                         int32_t* __restrict__ rank_offsets, int32_t* __restrict__ num_kept,
                         int32_t* __restrict__ slot_of, int32_t* __restrict__ perm_src,
                         int64_t send_rows) {
  pdl_trigger();  // the permute kernel may be scheduled now; it waits for this one
  count_pass(0, 1, idx, A, N, k, E, mode, chunk_hist, perm_src, send_rows);
  __syncthreads();
  scan_pass(chunk_hist, 1, E, R, rank_map, C, mode, expert_counts, kept_counts, expert_start,
            rank_counts, rank_offsets, num_kept);
  __syncthreads();
  assign_pass(0, idx, A, N, k, E, C, mode, chunk_hist, expert_start, num_kept, slot_of,
              perm_src);
}

// K3: one CTA walks tokens; each 16-byte vector of a row is loaded once and stored
// to every kept slot of that token.
constexpr int TP = 256;
constexpr int UNROLL = 4;

__global__ void __launch_bounds__(TP)
permute_kernel(const uint4* __restrict__ x, uint4* __restrict__ xperm,
               const int32_t* __restrict__ slot_of, int N, int k, int nvec) {
  pdl_wait();  // the assign pass has completed: the slots are final
  // a token's slots are loaded one token ahead, so the row copy does not wait on them;
  // a token whose every choice was dropped is not read at all
  int slots[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j)
    slots[j] = (j < k && blockIdx.x < N) ? slot_of[(int64_t)blockIdx.x * k + j] : -1;
  for (int t = blockIdx.x; t < N; t += gridDim.x) {
    const int tn = t + gridDim.x;
    int next[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) next[j] = (j < k && tn < N) ? slot_of[(int64_t)tn * k + j] : -1;
    bool any = false;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) any |= slots[j] >= 0;
    const uint4* src = x + (int64_t)t * nvec;
    if (!any) {
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) slots[j] = next[j];
      continue;
    }
    for (int v0 = threadIdx.x; v0 < nvec; v0 += TP * UNROLL) {
      uint4 buf[UNROLL];
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int v = v0 + u * TP;
        if (v < nvec) buf[u] = ld_stream_u4(src + v);
      }
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int v = v0 + u * TP;
        if (v < nvec) {
#pragma unroll
          for (int j = 0; j < kMaxTopK; ++j)
            if (slots[j] >= 0) xperm[(int64_t)slots[j] * nvec + v] = buf[u];
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) slots[j] = next[j];
  }
}

}  // namespace

cudaError_t launch_dispatch(const Cfg& c, const int32_t* topk_idx, const void* x, void* xperm,
                            int32_t* expert_counts, int32_t* kept_counts, int32_t* expert_start,
                            int32_t* rank_counts, int32_t* rank_offsets, int32_t* slot_of,
                            int32_t* perm_src, int32_t* num_kept, int32_t* chunk_hist,
                            cudaStream_t s) {
  if (c.n_chunks == 1) {
    count_scan_assign_kernel<<<1, T2, 0, s>>>(topk_idx, c.A, c.N, c.k, c.E, c.R, c.rank_map, c.C,
                                              c.mode, chunk_hist, expert_counts, kept_counts,
                                              expert_start, rank_counts, rank_offsets, num_kept,
                                              slot_of, perm_src, c.send_rows);
  } else {
    count_kernel<<<c.n_chunks, T2, 0, s>>>(topk_idx, c.A, c.N, c.k, c.E, c.mode, chunk_hist,
                                           perm_src, c.send_rows);
    scan_kernel<<<1, T2, 0, s>>>(chunk_hist, c.n_chunks, c.E, c.R, c.rank_map, c.C, c.mode,
                                 expert_counts, kept_counts, expert_start, rank_counts,
                                 rank_offsets, num_kept);
    assign_kernel<<<c.n_chunks, T2, 0, s>>>(topk_idx, c.A, c.N, c.k, c.E, c.C, c.mode,
                                            chunk_hist, expert_start, num_kept, slot_of,
                                            perm_src);
  }
  if (xperm) {
    const int nvec = (int)((int64_t)c.d * c.act_bytes / 16);
    int grid = num_sms() * 8;
    if (grid > c.N) grid = c.N;
    // a programmatic dependent of the assign pass
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_dependent(permute_kernel, dim3(grid), dim3(TP), 0, s,
                            static_cast<const uint4*>(x), static_cast<uint4*>(xperm),
                            static_cast<const int32_t*>(slot_of), c.N, c.k, nvec);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------- no-allocation variant
//
// For callers that cannot allocate device memory themselves.  The per-chunk expert
// histogram lives in one file-scope device array instead of the caller's workspace;
// every GPU that loads this library keeps it (kNoAllocHistInts int32 = 256 KiB) until
// the process exits.  Host code must not hand the array's name to a kernel (that is
// a host-side stand-in, not a device address): every call looks up its device
// address with the caller's device current.  The lookup is a host-side query, so a
// context that was destroyed and created again (a device reset) gets the new
// address on its next call instead of a stale one.
namespace {
static __device__ __align__(256) int32_t g_noalloc_hist[kNoAllocHistInts];
}  // namespace

cudaError_t launch_dispatch_noalloc(const Cfg& c, const int32_t* topk_idx, const void* x,
                                    void* xperm, int32_t* expert_counts, int32_t* kept_counts,
                                    int32_t* expert_start, int32_t* rank_counts,
                                    int32_t* rank_offsets, int32_t* slot_of, int32_t* perm_src,
                                    int32_t* num_kept, cudaStream_t s) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_hist);
  if (e != cudaSuccess) return e;
  // The count kernel writes every histogram entry that the scan and assign kernels
  // read later, so nothing left over from an earlier call is ever used.
  return launch_dispatch(c, topk_idx, x, xperm, expert_counts, kept_counts, expert_start,
                         rank_counts, rank_offsets, slot_of, perm_src, num_kept,
                         static_cast<int32_t*>(p), s);
}

}  // namespace moe
