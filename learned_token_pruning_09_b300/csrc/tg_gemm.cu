// Tensor-core GEMMs on tcgen05 with TMEM accumulators and TMA-fed shared
// memory stages, both run by CTA pairs (clusters of two CTAs on two SMs whose
// tensor cores execute one M=256 MMA together, cta_group::2):
//
//  * gate_kernel  -- TokenGate's gate MLP scorer (gate module: "an MLP scores
//    every token from its post-attention residual at layer L").  A pair of
//    CTAs takes 256 residual rows at a time; the pair's tensor cores compute
//    U = X W1^T (256 x h, fp32 in TMEM) and the epilogue fuses + b1,
//    exact-erf GELU, the 1-wide projection with w2, + b2 and logsigmoid,
//    writing one fp32 score per prunable row (document rows, or the rows of a
//    per-row mask) and 0 for every other row.
//  * linear_kernel -- out = A W^T (+ residual) in bf16, the per-layer Q/K/V and
//    output projections of the stacked long-context workload, 256 x 256 tiles.
//
// The shared scheme: each CTA stages its own 128 rows of the A operand and one
// half of the B operand's rows (the pair splits B), so the shared-memory
// traffic per SM is that of an M=128, N=128 MMA while the tensor cores run
// M=256, N=256; every copy of either CTA completes on the leader's (rank 0)
// stage barrier; the leader's MMA commits are multicast to both CTAs; the
// accumulators are double-buffered in TMEM so that the epilogue of one tile
// overlaps the MMAs of the next.
#include "tg_common.cuh"

namespace tg {

constexpr int kBM = 128;                   // rows of A per CTA
constexpr int kBK = 64;                    // one 128-byte swizzle row of bf16
constexpr uint32_t kPairABytes = kBM * kBK * 2;   // 16 KB: 128 rows of one K block
constexpr int kPairThreads = 256;
constexpr int kPairMaxStages = 8;

__host__ __device__ inline uint32_t tmem_cols_for(int n) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(n)) c <<= 1;
  return c;
}

// Barriers of a pair's stage ring and accumulators.  Placed after the ring in
// dynamic shared memory: the kernels have no static shared memory, so the
// ring starts at the 1024-byte aligned base and needs no alignment slack.
struct PairHead {
  uint64_t full[kPairMaxStages];        // leader: both CTAs' copies of a stage landed
  uint64_t empty[kPairMaxStages];       // the pair's MMAs are done with a stage
  uint64_t acc_full[2];                 // accumulator buffer complete
  uint64_t acc_empty[2];                // leader: both epilogues have read a buffer
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t peer_issued;                 // leader: stages the other CTA issued
  volatile int abort;
};

// Stages that fit the device's per-block shared memory next to `tail` bytes.
static cudaError_t pair_stages(size_t stage_bytes, size_t tail, int* n_st) {
  int dev = 0, max_smem = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  int n = static_cast<int>((static_cast<size_t>(max_smem) - tail) / stage_bytes);
  if (n > kPairMaxStages) n = kPairMaxStages;
  if (n < 2) return cudaErrorInvalidConfiguration;
  *n_st = n;
  return cudaSuccess;
}

// Barrier setup by thread 0 (the acc_empty count is one arrive per epilogue
// warp of both CTAs).
__device__ __forceinline__ void pair_init(PairHead& h, int n_st, int epi_warps) {
  for (int i = 0; i < n_st; ++i) { mbar_init(&h.full[i], 1); mbar_init(&h.empty[i], 1); }
  for (int b = 0; b < 2; ++b) { mbar_init(&h.acc_full[b], 1); mbar_init(&h.acc_empty[b], 2 * epi_warps); }
  mbar_init(&h.mma_done, 1);
  h.abort = 0;
  fence_barrier_init();
}

// Producer step: wait until stage `issued % n_st` is free, then copy this
// CTA's A rows and B half into it; both copies complete on the leader's
// barrier.  Returns false when the wait ran out (or another role aborted).
__device__ __forceinline__ bool pair_issue(PairHead& h, uint8_t* ring, uint32_t issued, uint32_t n_st,
                                           uint32_t stage_bytes, bool leader, uint32_t full0,
                                           const CUtensorMap* map_a, int ax, int ay,
                                           const CUtensorMap* map_b, int bx, int by,
                                           long long wd, unsigned int* status) {
  const uint32_t st = issued % n_st;
  const uint32_t use = issued / n_st;
  if (!mbar_wait(&h.empty[st], (use & 1u) ^ 1u, wd, status, kStatusTimeout) || h.abort) {
    h.abort = 1;
    return false;
  }
  uint8_t* s = ring + st * stage_bytes;
  if (leader) mbar_arrive_expect_tx(&h.full[st], 2 * stage_bytes);
  tma_load_2d_pair(s, map_a, full0 + st * 8u, ax, ay);
  tma_load_2d_pair(s + kPairABytes, map_b, full0 + st * 8u, bx, by);
  return true;
}

// The leader's MMAs of one K block (4 x K16 steps) into accumulator `d`.
__device__ __forceinline__ void pair_mma_kblock(uint32_t d, const uint8_t* stage, uint32_t idesc, bool first) {
  const uint32_t sa = smem_u32(stage);
  const uint32_t sb = sa + kPairABytes;
#pragma unroll
  for (int ks = 0; ks < kBK / 16; ++ks)
    mma_ss_pair(d, smem_desc_sw128(sa + ks * 32, 16, 1024), smem_desc_sw128(sb + ks * 32, 16, 1024), idesc,
                (!first || ks > 0) ? 1u : 0u);
}

// The leader's share of the final drain: every copy either CTA issued must
// land before the pair may leave.  The two producers stop together unless a
// wait ran out; then the leader settles the difference: it arrives for a
// stage only the other CTA issued, and counts off the other CTA's share of a
// stage it issued alone.  Called after a cluster barrier that follows the
// other CTA's store of its count.
__device__ __forceinline__ void pair_drain(PairHead& h, uint32_t own, uint32_t n_st, uint32_t stage_bytes,
                                           unsigned int* status) {
  const uint32_t peer = h.peer_issued;
  for (uint32_t g = own; g < peer; ++g) mbar_arrive_expect_tx(&h.full[g % n_st], stage_bytes);
  for (uint32_t g = peer; g < own; ++g) mbar_complete_tx(&h.full[g % n_st], stage_bytes);
  const uint32_t last_g = own > peer ? own : peer;
  for (uint32_t st = 0; st < n_st && st < last_g; ++st) {
    const uint32_t last = ((last_g - 1 - st) / n_st) * n_st + st;
    mbar_wait(&h.full[st], (last / n_st) & 1u, kDrainCycles, status, kStatusTimeout);
  }
}

// Launch a pair kernel on as many pairs as the device co-schedules, at most
// `units` (the persistent pairs take the units round-robin).
template <typename... Args>
static cudaError_t launch_pairs(void (*kernel)(Args...), size_t smem, long long units, cudaStream_t st,
                                int num_sms, Args... args) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2u * static_cast<unsigned>(num_sms / 2));
  int n_clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&n_clusters, kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (n_clusters < 1) return cudaErrorInvalidConfiguration;
  const long long pairs = units < n_clusters ? units : n_clusters;
  cfg.gridDim = dim3(2u * static_cast<unsigned>(pairs));
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---------------------------------------------------------------------------
// gate
// ---------------------------------------------------------------------------
// Pair q takes 256-row blocks q, q + P, q + 2P, ... (P pairs) and walks each
// block's K from a different starting point, so that the pairs do not all
// read the same W1 block from L2 at the same moment.  B = W1: each CTA stages
// W1 rows [rank h/2, rank h/2 + h/2).
//
// Warp roles (256 threads per CTA): warp 0 lane 0 issues this CTA's copies; in
// the leader warp 1 lane 0 issues the pair MMAs; warp 1 of each CTA takes part
// in the pair's TMEM allocation; warps 4-7 run the epilogue on the CTA's own
// 128 rows, one thread per row.
struct GateTail {
  PairHead head;
  alignas(16) float b1[256];
  alignas(16) float w2[256];
};

// Whether `row` is a document row; *seq = its sequence.
// the sequence of a row: the largest b with cu_seqlens[b] <= row
__device__ __forceinline__ int seq_of_row(const GateArgs& a, long long row) {
  int lo = 0, hi = a.batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.cu_seqlens + mid) <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ bool row_is_doc(const GateArgs& a, long long row, int* seq) {
  const int lo = seq_of_row(a, row);
  *seq = lo;
  const int start = __ldg(a.cu_seqlens + lo);
  const int nd = __ldg(a.n_doc + lo);
  const int len = __ldg(a.cu_seqlens + lo + 1) - start;
  if (nd < 0 || nd > len) {
    record_error(a.status, kStatusIndex);
    return false;
  }
  return row - start < nd;
}

__global__ void __launch_bounds__(kPairThreads, 1)
gate_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w1,
            GateArgs a, int n_st) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = smem_raw;
  const int hb = a.h / 2;                          // W1 rows staged by each CTA
  const uint32_t stage_bytes = kPairABytes + static_cast<uint32_t>(hb) * kBK * 2;
  GateTail& tail = *reinterpret_cast<GateTail*>(smem_raw + static_cast<size_t>(n_st) * stage_bytes);
  PairHead& head = tail.head;
  // 128-byte swizzled TMA and MMA tiles need a 1024-byte aligned ring; both
  // CTAs of a pair see the same base, so both leave here together
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) record_error(a.status, kStatusIndex);
    return;
  }
  const int warp = warp_id();
  const int lane = lane_id();
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const uint32_t half_cols = tmem_cols_for(a.h);   // one accumulator buffer
  const uint32_t ncols = 2 * half_cols;
  const long long n_blocks = (a.n_rows + 2 * kBM - 1) / (2 * kBM);   // 256-row blocks
  const int n_pairs = static_cast<int>(gridDim.x >> 1);
  const int q = static_cast<int>(blockIdx.x >> 1);
  const int n_pass = (q < n_blocks) ? static_cast<int>((n_blocks - q + n_pairs - 1) / n_pairs) : 0;
  const int nk = a.d / kBK;
  const long long wd = a.watchdog;

  if (threadIdx.x == 0) {
    pair_init(head, n_st, 4);
    prefetch_tmap(&map_x);
    prefetch_tmap(&map_w1);
  }
  if (warp == 1) { tmem_alloc_pair(&head.tmem_base, ncols); tmem_relinquish_pair(); }
  for (int i = threadIdx.x; i < a.h; i += kPairThreads) {
    tail.b1[i] = a.b1 ? a.b1[i] : 0.0f;
    tail.w2[i] = __bfloat162float(a.w2[i]);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();      // both CTAs' barriers exist before either signals the other
  tc_fence_after();

  // the top-K launched after the gate may start launching now (its CTAs wait
  // for the scores before they read anything)
  pdl_trigger();
  uint32_t issued = 0;                 // warp 0 lane 0: stages this CTA issued
  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer: this CTA's X rows and W1 half ----------------
    const uint32_t full0 = mapa_shared(smem_u32(&head.full[0]), 0);
    bool ok = true;
    for (int p = 0; p < n_pass && ok; ++p) {
      const long long blk = q + static_cast<long long>(p) * n_pairs;
      const int row0 = static_cast<int>(blk * 2 * kBM) + static_cast<int>(rank) * kBM;
      const int kb0 = (q + p) % nk;
      for (int i = 0; i < nk && ok; ++i) {
        int kb = kb0 + i;
        if (kb >= nk) kb -= nk;
        ok = pair_issue(head, ring, issued, n_st, stage_bytes, leader, full0, &map_x, kb * kBK, row0, &map_w1,
                        kb * kBK, static_cast<int>(rank) * hb, wd, a.status);
        if (ok) ++issued;
      }
    }
    if (!leader) st_cluster_u32(mapa_shared(smem_u32(&head.peer_issued), 0), issued);
  } else if (warp == 1 && lane == 0 && leader) {
    // ---------------- pair MMA issuer ----------------
    const uint32_t idesc = idesc_bf16_f32(2 * kBM, static_cast<uint32_t>(a.h), 0, 0);
    uint32_t g = 0;
    bool ok = true;
    for (int p = 0; p < n_pass && ok; ++p) {
      const int b = p & 1;
      // the epilogues of both CTAs must have read this buffer's previous block
      ok = mbar_wait(&head.acc_empty[b], ((static_cast<uint32_t>(p) >> 1) & 1u) ^ 1u, wd, a.status, kStatusTimeout) &&
           !head.abort;
      if (!ok) break;
      tc_fence_after();
      const uint32_t d = head.tmem_base + static_cast<uint32_t>(b) * half_cols;
      for (int i = 0; i < nk; ++i, ++g) {
        const int st = static_cast<int>(g % n_st);
        ok = mbar_wait(&head.full[st], (g / n_st) & 1u, wd, a.status, kStatusTimeout) && !head.abort;
        if (!ok) break;
        tc_fence_after();
        pair_mma_kblock(d, ring + st * stage_bytes, idesc, i == 0);
        mma_commit_pair_mc(&head.empty[st], 0x3);
      }
      if (ok) mma_commit_pair_mc(&head.acc_full[b], 0x3);
    }
    if (!ok) head.abort = 1;
    // every MMA must have finished before TMEM may be freed
    mma_commit_pair_mc(&head.mma_done, 0x1);
    mbar_wait(&head.mma_done, 0, kDrainCycles, a.status, kStatusTimeout);
  } else if (warp >= 4) {
    // ---------------- epilogue: + b1, GELU, . w2, + b2, logsigmoid ----------------
    const int sub = warp & 3;                               // TMEM lane quarter
    const uint32_t acc_empty0 = mapa_shared(smem_u32(&head.acc_empty[0]), 0);
    for (int p = 0; p < n_pass; ++p) {
      const int b = p & 1;
      const long long blk = q + static_cast<long long>(p) * n_pairs;
      const long long row = blk * 2 * kBM + static_cast<long long>(rank) * kBM + sub * 32 + lane;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&head.acc_full[b], (static_cast<uint32_t>(p) >> 1) & 1u, wd,
                                                         a.status, kStatusTimeout));
      if (!ok || head.abort) { head.abort = 1; break; }
      tc_fence_after();
      const uint32_t taddr = head.tmem_base + static_cast<uint32_t>(b) * half_cols +
                             (static_cast<uint32_t>(sub * 32) << 16);
      // Branch-free 32-column chunks (then one 16-column tail when h % 32 ==
      // 16) so the GELU chains of a chunk interleave; two partial sums.
      float2 zp[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
      const float2* b1p = reinterpret_cast<const float2*>(tail.b1);
      const float2* w2p = reinterpret_cast<const float2*>(tail.w2);
      int c0 = 0;
      for (; c0 + 32 <= a.h; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(taddr + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 u = __fadd2_rn(make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])),
                                      b1p[(c0 >> 1) + i]);
          zp[i & 1] = __ffma2_rn(w2p[(c0 >> 1) + i], gelu_erf2(u), zp[i & 1]);
        }
      }
      if (c0 < a.h) {
        uint32_t r[16];
        tmem_ld16(taddr + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 u = __fadd2_rn(make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])),
                                      b1p[(c0 >> 1) + i]);
          zp[i & 1] = __ffma2_rn(w2p[(c0 >> 1) + i], gelu_erf2(u), zp[i & 1]);
        }
      }
      float z = (zp[0].x + zp[0].y) + (zp[1].x + zp[1].y);
      // this warp is done with the buffer: tell the leader's MMA issuer
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty0 + static_cast<uint32_t>(b) * 8u);
      int seq = 0;
      bool counted = false;
      float sc = 0.0f;
      if (row < a.n_rows) {
        z += a.b2;
        // logsigmoid(z) = -log1p(exp(-z)) (z >= 0), z - log1p(exp(z)) (z < 0)
        sc = (z >= 0.0f) ? -log1pf(expf(-z)) : z - log1pf(expf(z));
        bool prun;
        if (a.prunable) {
          prun = __ldg(a.prunable + row) != 0;
          if (prun && a.hist) seq = seq_of_row(a, row);   // the histograms are per sequence
        } else {
          prun = row_is_doc(a, row, &seq);
        }
        a.s_out[row] = prun ? sc : 0.0f;
        counted = prun;
      }
      if (a.hist) {
        // the top-K's first two radix digits, counted here: the top 8 and the
        // top 16 bits of the score's order key, one atomic per distinct
        // (sequence, bin) of the warp
        const uint32_t key = order_key(sc);
        uint32_t* hs = a.hist + static_cast<long long>(seq) * kHistWords;
        const uint32_t ck = counted ? ((static_cast<uint32_t>(seq) << 8) | (key >> 24)) : 0xFFFFFFFFu;
        const uint32_t cm = __match_any_sync(0xffffffffu, ck);
        if (counted && lane == __ffs(cm) - 1) atomicAdd(hs + (key >> 24), static_cast<uint32_t>(__popc(cm)));
        const uint32_t fk = counted ? ((static_cast<uint32_t>(seq) << 16) | (key >> 16)) : 0xFFFFFFFFu;
        const uint32_t fm = __match_any_sync(0xffffffffu, fk);
        if (counted && lane == __ffs(fm) - 1)
          atomicAdd(hs + kHistCoarse + fine_slot(key >> 16), static_cast<uint32_t>(__popc(fm)));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();      // every role is done; the other CTA's issue count is in place
  if (leader && warp == 0 && lane == 0) pair_drain(head, issued, static_cast<uint32_t>(n_st), stage_bytes, a.status);
  __syncthreads();
  cluster_sync();      // no CTA leaves while the other may still signal it
  if (warp == 1) { tc_fence_after(); tmem_dealloc_pair(head.tmem_base, ncols); }
}

cudaError_t launch_gate(const CUtensorMap& map_x, const CUtensorMap& map_w1, const GateArgs& a,
                        cudaStream_t st) {
  if (a.n_rows == 0) return cudaSuccess;
  const size_t stage_bytes = kPairABytes + static_cast<size_t>(a.h / 2) * kBK * 2;
  int n_st = 0;
  cudaError_t e = pair_stages(stage_bytes, sizeof(GateTail), &n_st);
  if (e != cudaSuccess) return e;
  const size_t smem = static_cast<size_t>(n_st) * stage_bytes + sizeof(GateTail);
  const long long blocks = (a.n_rows + 2 * kBM - 1) / (2 * kBM);
  return launch_pairs(gate_kernel, smem, blocks, st, a.num_sms, map_x, map_w1, a, n_st);
}

// ---------------------------------------------------------------------------
// linear: out = A W^T (+ residual), bf16 out
// ---------------------------------------------------------------------------
// Tiles of 256 rows x bn columns (bn = 256, or n when smaller); pair q takes
// tiles q, q + P, ... in row-major tile order.  B = W: each CTA stages W rows
// [n0 + rank bn/2, + bn/2).  Epilogue: 4 warps per CTA, one thread per row,
// fp32 accumulators rounded once to bf16 after the residual add.
struct LinearTail {
  PairHead head;
};

// One row's share of the Q/K/V projection epilogue: the accumulator columns
// [n0, n0 + ncols) of buffer `tbase` (whole heads of head_dim), rotated by
// RoPE at the row's position when the head is a q or k head, rounded to bf16
// and written to q_out, k_out or v_out.  Rotate-half pairs column c with
// c + D/2 of the same head, so each step reads 32 columns of both halves of a
// head; the 32 angles of a step are shared by every head of the tile.  The
// warp's last TMEM read releases the buffer (acc_empty, on the leader).
__device__ __forceinline__ void qkv_rope_epilogue(const LinearArgs& a, uint32_t tbase, long long row, int n0,
                                                  int ncols, uint32_t acc_empty_addr, int lane) {
  const int D = a.head_dim, half = D >> 1;
  const int heads_here = ncols / D;
  const int head0 = n0 / D;
  const bool in_rows = row < a.m;
  const int p = in_rows ? __ldg(a.pos + row) : 0;
  const bool rot_tile = head0 < a.hq + a.hkv;         // the tile holds a q or k head
  for (int f0 = 0; f0 < half; f0 += 32) {
    float cs[32], sn[32];
    if (rot_tile) {
#pragma unroll
      for (int j = 0; j < 32; ++j) rope_sincos(p, a.freqs.turns_hi[f0 + j], a.freqs.turns_lo[f0 + j], &sn[j], &cs[j]);
    }
    for (int hh = 0; hh < heads_here; ++hh) {
      uint32_t rl[32], rh[32];
      tmem_ld32(tbase + static_cast<uint32_t>(hh * D + f0), rl);
      tmem_ld32(tbase + static_cast<uint32_t>(hh * D + f0 + half), rh);
      tmem_ld_wait();
      if (f0 + 32 >= half && hh + 1 == heads_here) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty_addr);
      }
      if (!in_rows) continue;
      const int head = head0 + hh;
      __nv_bfloat16* dst;
      bool rot = true;
      if (head < a.hq) {
        dst = static_cast<__nv_bfloat16*>(a.q_out) + (row * a.hq + head) * static_cast<long long>(D);
      } else if (head < a.hq + a.hkv) {
        dst = static_cast<__nv_bfloat16*>(a.k_out) + (row * a.hkv + (head - a.hq)) * static_cast<long long>(D);
      } else {
        dst = static_cast<__nv_bfloat16*>(a.v_out) +
              (row * a.hkv + (head - a.hq - a.hkv)) * static_cast<long long>(D);
        rot = false;
      }
      uint4 olo[4], ohi[4];
      uint32_t* pl = reinterpret_cast<uint32_t*>(olo);
      uint32_t* ph = reinterpret_cast<uint32_t*>(ohi);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float l0 = __uint_as_float(rl[2 * j]), l1 = __uint_as_float(rl[2 * j + 1]);
        const float h0 = __uint_as_float(rh[2 * j]), h1 = __uint_as_float(rh[2 * j + 1]);
        if (rot) {
          pl[j] = pack_bf16x2(l0 * cs[2 * j] - h0 * sn[2 * j], l1 * cs[2 * j + 1] - h1 * sn[2 * j + 1]);
          ph[j] = pack_bf16x2(h0 * cs[2 * j] + l0 * sn[2 * j], h1 * cs[2 * j + 1] + l1 * sn[2 * j + 1]);
        } else {
          pl[j] = pack_bf16x2(l0, l1);
          ph[j] = pack_bf16x2(h0, h1);
        }
      }
      uint4* dl = reinterpret_cast<uint4*>(dst + f0);
      uint4* dh = reinterpret_cast<uint4*>(dst + f0 + half);
#pragma unroll
      for (int v = 0; v < 4; ++v) { dl[v] = olo[v]; dh[v] = ohi[v]; }
    }
  }
}

template <bool kQkv>
__global__ void __launch_bounds__(kPairThreads, 1)
linear_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_w,
              LinearArgs a, int bn, int n_st) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = smem_raw;
  const uint32_t stage_bytes = kPairABytes + static_cast<uint32_t>(bn / 2) * kBK * 2;
  PairHead& head = reinterpret_cast<LinearTail*>(smem_raw + static_cast<size_t>(n_st) * stage_bytes)->head;
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) record_error(a.status, kStatusIndex);
    return;
  }
  const int warp = warp_id();
  const int lane = lane_id();
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const uint32_t half_cols = tmem_cols_for(bn);
  const uint32_t ncols = 2 * half_cols;
  const long long n_mt = (a.m + 2 * kBM - 1) / (2 * kBM);
  const int n_nt = (a.n + bn - 1) / bn;
  const long long n_tiles = n_mt * n_nt;
  const int n_pairs = static_cast<int>(gridDim.x >> 1);
  const int q = static_cast<int>(blockIdx.x >> 1);
  const int n_mine = (q < n_tiles) ? static_cast<int>((n_tiles - q + n_pairs - 1) / n_pairs) : 0;
  const int nk = a.kdim / kBK;
  const long long wd = a.watchdog;

  if (threadIdx.x == 0) {
    pair_init(head, n_st, 4);
    prefetch_tmap(&map_a);
    prefetch_tmap(&map_w);
  }
  if (warp == 1) { tmem_alloc_pair(&head.tmem_base, ncols); tmem_relinquish_pair(); }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();

  uint32_t issued = 0;
  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer: this CTA's A rows and W half ----------------
    const uint32_t full0 = mapa_shared(smem_u32(&head.full[0]), 0);
    bool ok = true;
    for (int p = 0; p < n_mine && ok; ++p) {
      const long long tile = q + static_cast<long long>(p) * n_pairs;
      const int m0 = static_cast<int>((tile / n_nt) * 2 * kBM) + static_cast<int>(rank) * kBM;
      const int n0 = static_cast<int>(tile % n_nt) * bn + static_cast<int>(rank) * (bn / 2);
      for (int kb = 0; kb < nk && ok; ++kb) {
        ok = pair_issue(head, ring, issued, n_st, stage_bytes, leader, full0, &map_a, kb * kBK, m0, &map_w,
                        kb * kBK, n0, wd, a.status);
        if (ok) ++issued;
      }
    }
    if (!leader) st_cluster_u32(mapa_shared(smem_u32(&head.peer_issued), 0), issued);
  } else if (warp == 1 && lane == 0 && leader) {
    // ---------------- pair MMA issuer ----------------
    const uint32_t idesc = idesc_bf16_f32(2 * kBM, static_cast<uint32_t>(bn), 0, 0);
    uint32_t g = 0;
    bool ok = true;
    for (int p = 0; p < n_mine && ok; ++p) {
      const int b = p & 1;
      ok = mbar_wait(&head.acc_empty[b], ((static_cast<uint32_t>(p) >> 1) & 1u) ^ 1u, wd, a.status, kStatusTimeout) &&
           !head.abort;
      if (!ok) break;
      tc_fence_after();
      const uint32_t d = head.tmem_base + static_cast<uint32_t>(b) * half_cols;
      for (int kb = 0; kb < nk; ++kb, ++g) {
        const int st = static_cast<int>(g % n_st);
        ok = mbar_wait(&head.full[st], (g / n_st) & 1u, wd, a.status, kStatusTimeout) && !head.abort;
        if (!ok) break;
        tc_fence_after();
        pair_mma_kblock(d, ring + st * stage_bytes, idesc, kb == 0);
        mma_commit_pair_mc(&head.empty[st], 0x3);
      }
      if (ok) mma_commit_pair_mc(&head.acc_full[b], 0x3);
    }
    if (!ok) head.abort = 1;
    mma_commit_pair_mc(&head.mma_done, 0x1);
    mbar_wait(&head.mma_done, 0, kDrainCycles, a.status, kStatusTimeout);
  } else if (warp >= 4) {
    // ---------------- epilogue: (+ residual), bf16 ----------------
    const int sub = warp & 3;
    const uint32_t acc_empty0 = mapa_shared(smem_u32(&head.acc_empty[0]), 0);
    for (int p = 0; p < n_mine; ++p) {
      const int b = p & 1;
      const long long tile = q + static_cast<long long>(p) * n_pairs;
      const long long row = (tile / n_nt) * 2 * kBM + static_cast<long long>(rank) * kBM + sub * 32 + lane;
      const int n0 = static_cast<int>(tile % n_nt) * bn;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&head.acc_full[b], (static_cast<uint32_t>(p) >> 1) & 1u, wd,
                                                         a.status, kStatusTimeout));
      if (!ok || head.abort) { head.abort = 1; break; }
      tc_fence_after();
      const uint32_t tbase = head.tmem_base + static_cast<uint32_t>(b) * half_cols +
                             (static_cast<uint32_t>(sub * 32) << 16);
      const int ncols_here = min(bn, a.n - n0);
      if constexpr (kQkv) {
        qkv_rope_epilogue(a, tbase, row, n0, ncols_here, acc_empty0 + static_cast<uint32_t>(b) * 8u, lane);
      } else {
        for (int c0 = 0; c0 < ncols_here; c0 += 32) {
          uint32_t r[32];
          const bool full32 = ncols_here - c0 >= 32;
          if (full32) {
            tmem_ld32(tbase + c0, r);
          } else {
            uint32_t r16[16];
            tmem_ld16(tbase + c0, r16);
#pragma unroll
            for (int i = 0; i < 16; ++i) { r[i] = r16[i]; r[16 + i] = 0u; }
          }
          tmem_ld_wait();
          if (c0 + 32 >= ncols_here) {
            // the last TMEM read of this buffer: tell the leader's MMA issuer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc_empty0 + static_cast<uint32_t>(b) * 8u);
          }
          if (row < a.m) {
            const size_t off = static_cast<size_t>(row) * a.n + n0 + c0;
            const int nv = full32 ? 4 : 2;              // 16-byte vectors (8 bf16)
            uint4 res[4] = {};
            if (a.residual) {
              const uint4* rp = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.residual) + off);
              for (int v = 0; v < nv; ++v) res[v] = rp[v];
            }
            uint4* op = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + off);
            for (int v = 0; v < nv; ++v) {
              const __nv_bfloat162* rb = reinterpret_cast<const __nv_bfloat162*>(&res[v]);
              uint4 o;
              uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float x0 = __uint_as_float(r[v * 8 + 2 * e]);
                float x1 = __uint_as_float(r[v * 8 + 2 * e + 1]);
                if (a.residual) {
                  const float2 rr = __bfloat1622float2(rb[e]);
                  x0 += rr.x;
                  x1 += rr.y;
                }
                ow[e] = pack_bf16x2(x0, x1);
              }
              op[v] = o;
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (leader && warp == 0 && lane == 0) pair_drain(head, issued, static_cast<uint32_t>(n_st), stage_bytes, a.status);
  __syncthreads();
  cluster_sync();
  if (warp == 1) { tc_fence_after(); tmem_dealloc_pair(head.tmem_base, ncols); }
}

cudaError_t launch_linear(const CUtensorMap& map_a, const CUtensorMap& map_w, const LinearArgs& a,
                          cudaStream_t st) {
  if (a.m == 0 || a.n == 0) return cudaSuccess;
  const int bn = linear_tile_n(a.n);
  const size_t stage_bytes = kPairABytes + static_cast<size_t>(bn / 2) * kBK * 2;
  int n_st = 0;
  cudaError_t e = pair_stages(stage_bytes, sizeof(LinearTail), &n_st);
  if (e != cudaSuccess) return e;
  const size_t smem = static_cast<size_t>(n_st) * stage_bytes + sizeof(LinearTail);
  const long long tiles = ((a.m + 2 * kBM - 1) / (2 * kBM)) * ((a.n + bn - 1) / bn);
  if (a.q_out) return launch_pairs(linear_kernel<true>, smem, tiles, st, a.num_sms, map_a, map_w, a, bn, n_st);
  return launch_pairs(linear_kernel<false>, smem, tiles, st, a.num_sms, map_a, map_w, a, bn, n_st);
}

}  // namespace tg
