// Tensor-core GEMMs on tcgen05 with TMEM accumulators and TMA-fed shared
// memory stages:
//
//  * gate_kernel  -- TokenGate's gate MLP scorer (gate module: "an MLP scores
//    every token from its post-attention residual at layer L").  One CTA
//    takes 128 residual rows; the tensor cores compute U = X W1^T (128 x h,
//    fp32 in TMEM) and the epilogue fuses + b1, exact-erf GELU, the 1-wide
//    projection with w2, + b2 and logsigmoid, writing one fp32 score per row
//    (0 for question rows).
//  * linear_kernel -- out = A W^T (+ residual) in bf16, the per-layer Q/K/V and
//    output projections of the stacked long-context workload.
//
// Warp roles (192 threads): warp 0 issues TMA loads, warp 1 allocates TMEM
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
// Persistent: one CTA per SM.  The residual rows are cut into 128-row blocks;
// CTA c owns blocks c, c + G, c + 2G, ... (G CTAs) and takes them two at a
// time.  The two blocks of a pass accumulate into two TMEM accumulators and
// share every W1 stage, which halves the W1 reads from L2 compared with one
// block per pass; a CTA left with one block runs a half pass.  Each pass
// walks its K blocks from a different starting block so that the CTAs do not
// all read the same W1 block at the same moment.  The epilogue (8 warps:
// warps 4-7 take the first block, warps 8-11 the second) releases TMEM
// before its final transform and store, so the next pass's MMAs start while
// it finishes; the producer runs ahead across passes.
constexpr int kGateThreads = 384;
constexpr int kGateM = 256;
constexpr int kGateMaxStages = 8;
constexpr int kGateATileBytes = kGateM * kBK * 2;   // 32 KB
constexpr int kGateSmemBudget = 200 * 1024;

struct GateSmemHead {
  uint64_t a_full[kGateMaxStages];
  uint64_t a_empty[kGateMaxStages];
  uint64_t b_full[kGateMaxStages];
  uint64_t b_empty[kGateMaxStages];
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t mma_done;
  uint32_t tmem_base;
  volatile int abort;
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
            GateArgs a, int n_a, int n_b) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ GateSmemHead head;
  __shared__ __align__(16) float sb1[256];
  __shared__ __align__(16) float sw2[256];
  // two rings: residual rows (from HBM, deeper) and W1 (L2-resident)
  uint8_t* ring_a = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = warp_id();
  const int lane = lane_id();
  const uint32_t half_cols = tmem_cols_for(a.h);
  const uint32_t ncols = 2 * half_cols;
  const int n_blocks = static_cast<int>((a.n_rows + kBM - 1) / kBM);
  const int G = gridDim.x;
  const int c = blockIdx.x;
  // pass p of this CTA covers blocks c + 2pG and c + (2p+1)G (if it exists)
  const int n_pass = (n_blocks - c + 2 * G - 1) / (2 * G);
  const int nk = a.d / kBK;
  const uint32_t b_bytes = static_cast<uint32_t>(a.h) * kBK * 2;
  uint8_t* ring_b = ring_a + static_cast<size_t>(n_a) * kGateATileBytes;
  const long long wd = a.watchdog;

  if (threadIdx.x == 0) {
    for (int i = 0; i < n_a; ++i) { mbar_init(&head.a_full[i], 1); mbar_init(&head.a_empty[i], 1); }
    for (int i = 0; i < n_b; ++i) { mbar_init(&head.b_full[i], 1); mbar_init(&head.b_empty[i], 1); }
    mbar_init(&head.acc_full, 1);
    mbar_init(&head.acc_empty, 256);
    mbar_init(&head.mma_done, 1);
    head.abort = 0;
    fence_barrier_init();
    prefetch_tmap(&map_x);
    prefetch_tmap(&map_w1);
  }
  if (warp == 1) { tmem_alloc(&head.tmem_base, ncols); tmem_relinquish(); }
  for (int i = threadIdx.x; i < a.h; i += kGateThreads) {
    sb1[i] = a.b1 ? a.b1[i] : 0.0f;
    sw2[i] = __bfloat162float(a.w2[i]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if ((warp == 0 || warp == 2) && lane == 0) {
    // ---------------- TMA producers: warp 0 residual rows, warp 2 W1 ----------------
    const bool rows = warp == 0;
    const int n_st = rows ? n_a : n_b;
    uint64_t* full = rows ? head.a_full : head.b_full;
    uint64_t* empty = rows ? head.a_empty : head.b_empty;
    uint32_t g = 0;                 // k blocks issued (the rings run across passes)
    for (int p = 0; p < n_pass && !head.abort; ++p) {
      const int blk0 = c + 2 * p * G;
      const int blk1 = blk0 + G;
      const bool has1 = blk1 < n_blocks;
      const int kb0 = (c + p) % nk;
      for (int i = 0; i < nk; ++i) {
        int kb = kb0 + i;
        if (kb >= nk) kb -= nk;
        const int st = static_cast<int>(g % n_st);
        const uint32_t use = g / n_st;
        if (!mbar_wait(&empty[st], (use & 1u) ^ 1u, wd, a.status, kStatusTimeout) || head.abort) {
          head.abort = 1;
          break;
        }
        if (rows) {
          uint8_t* sa = ring_a + st * kGateATileBytes;
          mbar_arrive_expect_tx(&full[st], (has1 ? 2u : 1u) * kATileBytes);
          tma_load_2d(sa, &map_x, &full[st], kb * kBK, blk0 * kBM);
          if (has1) tma_load_2d(sa + kATileBytes, &map_x, &full[st], kb * kBK, blk1 * kBM);
        } else {
          mbar_arrive_expect_tx(&full[st], b_bytes);
          tma_load_2d(ring_b + st * b_bytes, &map_w1, &full[st], kb * kBK, 0);
        }
        ++g;
      }
    }
    // the last copies into every stage must land before the CTA may leave
    for (uint32_t st = 0; st < static_cast<uint32_t>(n_st) && st < g; ++st) {
      const uint32_t last = ((g - 1 - st) / n_st) * n_st + st;
      mbar_wait(&full[st], (last / n_st) & 1u, kDrainCycles, a.status, kStatusTimeout);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kBM, static_cast<uint32_t>(a.h), 0, 0);
      const uint32_t acc0 = head.tmem_base;
      const uint32_t acc1 = head.tmem_base + half_cols;
      uint32_t g = 0;
      for (int it = 0; it < n_pass && !head.abort; ++it) {
        const bool has1 = c + (2 * it + 1) * G < n_blocks;
        // the epilogue must have read the previous pass's accumulators
        if (!mbar_wait(&head.acc_empty, (static_cast<uint32_t>(it) & 1u) ^ 1u, wd, a.status, kStatusTimeout)) {
          head.abort = 1;
          break;
        }
        tc_fence_after();
        bool ok = true;
        for (int i = 0; i < nk; ++i, ++g) {
          const int sa_i = static_cast<int>(g % n_a);
          const int sb_i = static_cast<int>(g % n_b);
          if (!mbar_wait(&head.a_full[sa_i], (g / n_a) & 1u, wd, a.status, kStatusTimeout) ||
              !mbar_wait(&head.b_full[sb_i], (g / n_b) & 1u, wd, a.status, kStatusTimeout) || head.abort) {
            head.abort = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(ring_a + sa_i * kGateATileBytes);
          const uint32_t sb = smem_u32(ring_b + sb_i * b_bytes);
#pragma unroll
          for (int ks = 0; ks < kBK / 16; ++ks) {
            const uint64_t db = smem_desc_sw128(sb + ks * 32, 16, 1024);
            const uint32_t acc = (i > 0 || ks > 0) ? 1u : 0u;
            mma_ss(acc0, smem_desc_sw128(sa + ks * 32, 16, 1024), db, idesc, acc);
            if (has1) mma_ss(acc1, smem_desc_sw128(sa + kATileBytes + ks * 32, 16, 1024), db, idesc, acc);
          }
          mma_commit(&head.a_empty[sa_i]);
          mma_commit(&head.b_empty[sb_i]);
        }
        mma_commit(&head.acc_full);
        if (!ok) break;
      }
      // every MMA must have finished before TMEM may be freed
      mma_commit(&head.mma_done);
      mbar_wait(&head.mma_done, 0, kDrainCycles, a.status, kStatusTimeout);
    }
  } else if (warp >= 4) {
    // ---------------- epilogue: + b1, GELU, . w2, + b2, logsigmoid ----------------
    const int half = (warp - 4) >> 2;
    const int sub = warp & 3;                               // TMEM lane quarter
    const uint32_t taddr = head.tmem_base + half * half_cols + (static_cast<uint32_t>(sub * 32) << 16);
    for (int it = 0; it < n_pass; ++it) {
      const int blk = c + (2 * it + half) * G;
      const long long row = static_cast<long long>(blk) * kBM + sub * 32 + lane;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&head.acc_full, static_cast<uint32_t>(it) & 1u, wd,
                                                         a.status, kStatusTimeout));
      if (!ok || head.abort) { head.abort = 1; break; }
      tc_fence_after();
      // Branch-free 32-column chunks (then one 16-column tail when h % 32 ==
      // 16) so the GELU chains of a chunk interleave; four partial sums.
      float2 zp[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
      const float2* b1p = reinterpret_cast<const float2*>(sb1);
      const float2* w2p = reinterpret_cast<const float2*>(sw2);
      if (blk < n_blocks) {
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
      }
      float z = (zp[0].x + zp[0].y) + (zp[1].x + zp[1].y);
      tc_fence_before();
      mbar_arrive(&head.acc_empty);      // accumulators may be overwritten now
      if (blk < n_blocks && row < a.n_rows) {
        z += a.b2;
        // logsigmoid(z) = -log1p(exp(-z)) (z >= 0), z - log1p(exp(z)) (z < 0)
        const float sc = (z >= 0.0f) ? -log1pf(expf(-z)) : z - log1pf(expf(z));
        a.s_out[row] = row_is_doc(a, row) ? sc : 0.0f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) { tc_fence_after(); tmem_dealloc(head.tmem_base, ncols); }
}

cudaError_t launch_gate(const CUtensorMap& map_x, const CUtensorMap& map_w1, const GateArgs& a,
                        cudaStream_t st) {
  if (a.n_rows == 0) return cudaSuccess;
  // W1 stages come from L2 (two suffice); the rest of the budget holds
  // residual-row stages, which come from HBM
  const size_t b_bytes = static_cast<size_t>(a.h) * kBK * 2;
  const int n_b = 2;
  int n_a = static_cast<int>((kGateSmemBudget - n_b * b_bytes) / kGateATileBytes);
  if (n_a > kGateMaxStages) n_a = kGateMaxStages;
  const size_t smem = 1024 + static_cast<size_t>(n_a) * kGateATileBytes + n_b * b_bytes;
  cudaError_t e = cudaFuncSetAttribute(gate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long blocks = (a.n_rows + kBM - 1) / kBM;
  const unsigned grid = static_cast<unsigned>(blocks < a.num_sms ? blocks : a.num_sms);
  gate_kernel<<<grid, kGateThreads, smem, st>>>(map_x, map_w1, a, n_a, n_b);
  return cudaGetLastError();
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
