// Tensor-core GEMMs on tcgen05 with TMEM accumulators and TMA-fed shared
// memory stages:
//
//  * gate_kernel  -- TokenGate's gate MLP scorer (gate module: "an MLP scores
//    every token from its post-attention residual at layer L").  A pair of
//    CTAs takes 256 residual rows at a time; the pair's tensor cores compute
//    U = X W1^T (256 x h, fp32 in TMEM) and the epilogue fuses + b1,
//    exact-erf GELU, the 1-wide projection with w2, + b2 and logsigmoid,
//    writing one fp32 score per row (0 for question rows).
//  * linear_kernel -- out = A W^T (+ residual) in bf16, the per-layer Q/K/V and
//    output projections of the stacked long-context workload.
//
// linear_kernel's warp roles (192 threads): warp 0 issues TMA loads, warp 1 allocates TMEM
// and issues the MMAs (one elected lane), warps 2..5 run the epilogue, one
// thread per accumulator row (warp w reads TMEM lanes 32*(w%4)..+31).
#include "tg_common.cuh"

namespace tg {

constexpr int kGemmThreads = 192;
constexpr int kBM = 128;
constexpr int kBK = 64;                    // one 128-byte swizzle row of bf16
constexpr int kATileBytes = kBM * kBK * 2; // 16 KB

struct GemmSmemHead {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t acc_full;
  uint32_t tmem_base;
  volatile int abort;
};

// Shared by both kernels: TMA producer + MMA issuer over the K dimension.
// A rows [m0, m0+128), B rows [n0, n0+bn), K = kdim.  Accumulates into TMEM
// columns [0, bn).  Returns (in every thread) after the roles are done with
// the mainloop; epilogue threads then wait on head->acc_full.
template <int kStages>
__device__ __forceinline__ void gemm_mainloop(const CUtensorMap* map_a, const CUtensorMap* map_b,
                                              GemmSmemHead* head, uint8_t* stages, int bn,
                                              int m0, int n0, int kdim, unsigned int* status,
                                              long long watchdog) {
  const int warp = warp_id();
  const int lane = lane_id();
  const int nk = kdim / kBK;
  const uint32_t b_bytes = static_cast<uint32_t>(bn) * kBK * 2;
  const uint32_t stage_bytes = kATileBytes + b_bytes;
  if (warp == 0 && lane == 0) {
    int issued = 0;
    for (int kb = 0; kb < nk; ++kb) {
      const int st = kb % kStages;
      const uint32_t use = kb / kStages;
      if (!mbar_wait(&head->empty[st], (use & 1u) ^ 1u, watchdog, status, kStatusTimeout)) {
        head->abort = 1;
        break;
      }
      if (head->abort) break;
      uint8_t* sa = stages + st * stage_bytes;
      mbar_arrive_expect_tx(&head->full[st], stage_bytes);
      tma_load_2d(sa, map_a, &head->full[st], kb * kBK, m0);
      tma_load_2d(sa + kATileBytes, map_b, &head->full[st], kb * kBK, n0);
      issued = kb + 1;
    }
    // wait for the last loads of every stage to land before anyone may leave
    for (int st = 0; st < kStages && st < issued; ++st) {
      const int last = ((issued - 1 - st) / kStages) * kStages + st;
      mbar_wait(&head->full[st], (static_cast<uint32_t>(last / kStages)) & 1u, kDrainCycles, status, kStatusTimeout);
    }
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_bf16_f32(kBM, static_cast<uint32_t>(bn), 0, 0);
    const uint32_t d_tmem = head->tmem_base;
    bool ok = true;
    for (int kb = 0; kb < nk && ok; ++kb) {
      const int st = kb % kStages;
      const uint32_t use = kb / kStages;
      if (!mbar_wait(&head->full[st], use & 1u, watchdog, status, kStatusTimeout) || head->abort) {
        head->abort = 1;
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sa = smem_u32(stages + st * stage_bytes);
      const uint32_t sb = sa + kATileBytes;
#pragma unroll
      for (int ks = 0; ks < kBK / 16; ++ks) {
        const uint64_t da = smem_desc_sw128(sa + ks * 32, 16, 1024);
        const uint64_t db = smem_desc_sw128(sb + ks * 32, 16, 1024);
        mma_ss(d_tmem, da, db, idesc, (kb > 0 || ks > 0) ? 1u : 0u);
      }
      mma_commit(&head->empty[st]);
    }
    mma_commit(&head->acc_full);
    // every MMA must have finished before TMEM may be freed
    mbar_wait(&head->acc_full, 0, kDrainCycles, status, kStatusTimeout);
  }
}

template <int kStages>
__device__ __forceinline__ size_t gemm_smem_bytes(int bn) {
  return 1024 + static_cast<size_t>(kStages) * (kATileBytes + bn * kBK * 2);
}

__host__ __device__ inline uint32_t tmem_cols_for(int n) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(n)) c <<= 1;
  return c;
}

// ---------------------------------------------------------------------------
// gate
// ---------------------------------------------------------------------------
// CTA pairs (clusters of two CTAs, one per SM): the two tensor cores of a pair
// compute U = X W1^T for 256 residual rows at a time with M=256 pair MMAs.
// Each CTA stages its own 128 rows of X and one half of W1's h rows (the B
// operand is split across the pair), which halves the shared-memory traffic
// per SM compared with one SM holding all of W1.  The accumulators (h fp32
// columns per row) are double-buffered in TMEM, so that the epilogue of one
// 256-row block runs while the MMAs of the next one fill the other buffer.
// Pair q takes blocks q, q + P, q + 2P, ... (P pairs) and walks each block's K
// from a different starting point, so that the pairs do not all read the same
// W1 block from L2 at the same moment.
//
// Warp roles (256 threads per CTA): warp 0 lane 0 issues this CTA's TMA loads,
// whose completion both CTAs count on the leader's (rank 0) stage barrier; in
// the leader warp 1 lane 0 issues the pair MMAs; warp 1 of each CTA takes part
// in the pair's TMEM allocation; warps 4-7 run the epilogue on the CTA's own
// 128 rows, one thread per row.
constexpr int kGateThreads = 256;
constexpr int kGateMaxStages = 8;
constexpr uint32_t kGateXBytes = kBM * kBK * 2;     // 16 KB: 128 rows of one K block

struct GateSmemHead {
  uint64_t full[kGateMaxStages];        // leader: both CTAs' copies of a stage landed
  uint64_t empty[kGateMaxStages];       // the pair's MMAs are done with a stage
  uint64_t acc_full[2];                 // accumulator buffer complete
  uint64_t acc_empty[2];                // leader: both epilogues have read a buffer
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t peer_issued;                 // leader: stages the other CTA issued
  volatile int abort;
};

// Placed after the stage ring in dynamic shared memory (the kernel has no
// static shared memory, so the ring starts at the 1024-byte aligned base and
// needs no alignment slack: one more stage fits).
struct GateSmemTail {
  GateSmemHead head;
  alignas(16) float b1[256];
  alignas(16) float w2[256];
};

__device__ __forceinline__ bool row_is_doc(const GateArgs& a, long long row) {
  int lo = 0, hi = a.batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.cu_seqlens + mid) <= row) lo = mid; else hi = mid - 1;
  }
  const int start = __ldg(a.cu_seqlens + lo);
  const int nd = __ldg(a.n_doc + lo);
  const int len = __ldg(a.cu_seqlens + lo + 1) - start;
  if (nd < 0 || nd > len) {
    record_error(a.status, kStatusIndex);
    return false;
  }
  return row - start < nd;
}

__global__ void __launch_bounds__(kGateThreads, 1)
gate_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w1,
            GateArgs a, int n_st) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = smem_raw;
  const int lane = lane_id();
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const uint32_t half_cols = tmem_cols_for(a.h);   // one accumulator buffer
  const uint32_t ncols = 2 * half_cols;
  const int hb = a.h / 2;                          // W1 rows staged by each CTA
  const uint32_t stage_bytes = kGateXBytes + static_cast<uint32_t>(hb) * kBK * 2;
  GateSmemTail& tail = *reinterpret_cast<GateSmemTail*>(smem_raw + static_cast<size_t>(n_st) * stage_bytes);
  GateSmemHead& head = tail.head;
  float* sb1 = tail.b1;
  float* sw2 = tail.w2;
  // 128-byte swizzled TMA and MMA tiles need a 1024-byte aligned ring; both
  // CTAs of a pair see the same base, so both leave here together
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) record_error(a.status, kStatusIndex);
    return;
  }
  const int warp = warp_id();  const long long n_blocks = (a.n_rows + 2 * kBM - 1) / (2 * kBM);   // 256-row blocks
  const int n_pairs = static_cast<int>(gridDim.x >> 1);
  const int q = static_cast<int>(blockIdx.x >> 1);
  const int n_pass = (q < n_blocks) ? static_cast<int>((n_blocks - q + n_pairs - 1) / n_pairs) : 0;
  const int nk = a.d / kBK;
  const long long wd = a.watchdog;

  if (threadIdx.x == 0) {
    for (int i = 0; i < n_st; ++i) {
      mbar_init(&head.full[i], 1);
      mbar_init(&head.empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&head.acc_full[b], 1);
      mbar_init(&head.acc_empty[b], 2 * 4);   // one arrive per epilogue warp of both CTAs
    }
    mbar_init(&head.mma_done, 1);
    head.abort = 0;
    fence_barrier_init();
    prefetch_tmap(&map_x);
    prefetch_tmap(&map_w1);
  }
  if (warp == 1) { tmem_alloc_pair(&head.tmem_base, ncols); tmem_relinquish_pair(); }
  for (int i = threadIdx.x; i < a.h; i += kGateThreads) {
    sb1[i] = a.b1 ? a.b1[i] : 0.0f;
    sw2[i] = __bfloat162float(a.w2[i]);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();      // both CTAs' barriers exist before either signals the other
  tc_fence_after();

  uint32_t issued = 0;                 // warp 0 lane 0: stages this CTA issued
  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer: this CTA's X rows and W1 half ----------------
    const uint32_t full0 = mapa_shared(smem_u32(&head.full[0]), 0);
    for (int p = 0; p < n_pass && !head.abort; ++p) {
      const long long blk = q + static_cast<long long>(p) * n_pairs;
      const int row0 = static_cast<int>(blk * 2 * kBM) + static_cast<int>(rank) * kBM;
      const int kb0 = (q + p) % nk;
      for (int i = 0; i < nk; ++i) {
        int kb = kb0 + i;
        if (kb >= nk) kb -= nk;
        const int st = static_cast<int>(issued % n_st);
        const uint32_t use = issued / n_st;
        if (!mbar_wait(&head.empty[st], (use & 1u) ^ 1u, wd, a.status, kStatusTimeout) || head.abort) {
          head.abort = 1;
          break;
        }
        uint8_t* s = ring + st * stage_bytes;
        if (leader) mbar_arrive_expect_tx(&head.full[st], 2 * stage_bytes);
        tma_load_2d_pair(s, &map_x, full0 + st * 8u, kb * kBK, row0);
        tma_load_2d_pair(s + kGateXBytes, &map_w1, full0 + st * 8u, kb * kBK, static_cast<int>(rank) * hb);
        ++issued;
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
        const uint32_t par = (g / n_st) & 1u;
        ok = mbar_wait(&head.full[st], par, wd, a.status, kStatusTimeout) && !head.abort;
        if (!ok) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(ring + st * stage_bytes);
        const uint32_t sb = sa + kGateXBytes;
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks)
          mma_ss_pair(d, smem_desc_sw128(sa + ks * 32, 16, 1024), smem_desc_sw128(sb + ks * 32, 16, 1024), idesc,
                      (i > 0 || ks > 0) ? 1u : 0u);
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
      const float2* b1p = reinterpret_cast<const float2*>(sb1);
      const float2* w2p = reinterpret_cast<const float2*>(sw2);
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
      if (row < a.n_rows) {
        z += a.b2;
        // logsigmoid(z) = -log1p(exp(-z)) (z >= 0), z - log1p(exp(z)) (z < 0)
        const float sc = (z >= 0.0f) ? -log1pf(expf(-z)) : z - log1pf(expf(z));
        a.s_out[row] = row_is_doc(a, row) ? sc : 0.0f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();      // every role is done; the other CTA's issue count is in place
  if (leader && warp == 0 && lane == 0) {
    // Every copy either CTA issued must land before the pair may leave.  The
    // two producers stop together unless a wait ran out; then the leader
    // settles the difference: it arrives for a stage only the other CTA
    // issued, and counts off the other CTA's share of a stage it issued alone.
    const uint32_t peer = head.peer_issued;
    for (uint32_t g = issued; g < peer; ++g) mbar_arrive_expect_tx(&head.full[g % n_st], stage_bytes);
    for (uint32_t g = peer; g < issued; ++g) mbar_complete_tx(&head.full[g % n_st], stage_bytes);
    const uint32_t last_g = issued > peer ? issued : peer;
    for (uint32_t st = 0; st < static_cast<uint32_t>(n_st) && st < last_g; ++st) {
      const uint32_t last = ((last_g - 1 - st) / n_st) * n_st + st;
      mbar_wait(&head.full[st], (last / n_st) & 1u, kDrainCycles, a.status, kStatusTimeout);
    }
  }
  __syncthreads();
  cluster_sync();      // no CTA leaves while the other may still signal it
  if (warp == 1) { tc_fence_after(); tmem_dealloc_pair(head.tmem_base, ncols); }
}

cudaError_t launch_gate(const CUtensorMap& map_x, const CUtensorMap& map_w1, const GateArgs& a,
                        cudaStream_t st) {
  if (a.n_rows == 0) return cudaSuccess;
  const size_t stage_bytes = kGateXBytes + static_cast<size_t>(a.h / 2) * kBK * 2;
  int dev = 0, max_smem = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  int n_st = static_cast<int>((static_cast<size_t>(max_smem) - sizeof(GateSmemTail)) / stage_bytes);
  if (n_st > kGateMaxStages) n_st = kGateMaxStages;
  if (n_st < 2) return cudaErrorInvalidConfiguration;
  const size_t smem = static_cast<size_t>(n_st) * stage_bytes + sizeof(GateSmemTail);
  e = cudaFuncSetAttribute(gate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long blocks = (a.n_rows + 2 * kBM - 1) / (2 * kBM);
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kGateThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // one pair per two SMs at most; a persistent pair takes several blocks
  cfg.gridDim = dim3(2u * static_cast<unsigned>(a.num_sms / 2));
  int n_clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&n_clusters, gate_kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (n_clusters < 1) return cudaErrorInvalidConfiguration;
  const long long pairs = blocks < n_clusters ? blocks : n_clusters;
  cfg.gridDim = dim3(2u * static_cast<unsigned>(pairs));
  return cudaLaunchKernelEx(&cfg, gate_kernel, map_x, map_w1, a, n_st);
}

// ---------------------------------------------------------------------------
// linear: out = A W^T (+ residual), bf16 out
// ---------------------------------------------------------------------------
constexpr int kLinStages = 4;
constexpr int kLinBN = 256;

__global__ void __launch_bounds__(kGemmThreads, 1)
linear_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_w,
              LinearArgs a, int bn) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ GemmSmemHead head;
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = warp_id();
  const int lane = lane_id();
  const int m0 = blockIdx.x * kBM;
  const int n0 = blockIdx.y * bn;
  const uint32_t ncols = tmem_cols_for(bn);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kLinStages; ++i) { mbar_init(&head.full[i], 1); mbar_init(&head.empty[i], 1); }
    mbar_init(&head.acc_full, 1);
    head.abort = 0;
    fence_barrier_init();
    prefetch_tmap(&map_a);
    prefetch_tmap(&map_w);
  }
  if (warp == 1) { tmem_alloc(&head.tmem_base, ncols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  gemm_mainloop<kLinStages>(&map_a, &map_w, &head, stages, bn, m0, n0, a.kdim, a.status, a.watchdog);

  if (warp >= 2) {
    const int sub = warp & 3;
    const long long row = m0 + sub * 32 + lane;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&head.acc_full, 0, a.watchdog, a.status, kStatusTimeout));
    tc_fence_after();
    const uint32_t tbase = head.tmem_base + (static_cast<uint32_t>(sub * 32) << 16);
    if (ok) {
      const int ncols_here = min(bn, a.n - n0);
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
  tc_fence_before();
  __syncthreads();
  if (warp == 1) { tc_fence_after(); tmem_dealloc(head.tmem_base, ncols); }
}

cudaError_t launch_linear(const CUtensorMap& map_a, const CUtensorMap& map_w, const LinearArgs& a,
                          cudaStream_t st) {
  if (a.m == 0 || a.n == 0) return cudaSuccess;
  const int bn = a.n >= kLinBN ? kLinBN : a.n;
  const size_t smem = 1024 + static_cast<size_t>(kLinStages) * (kATileBytes + bn * kBK * 2);
  cudaError_t e = cudaFuncSetAttribute(linear_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>((a.m + kBM - 1) / kBM), static_cast<unsigned>((a.n + bn - 1) / bn));
  linear_kernel<<<grid, kGemmThreads, smem, st>>>(map_a, map_w, a, bn);
  return cudaGetLastError();
}

}  // namespace tg
