// Token-gated causal attention over the kept tokens (TokenGate, "What is
// token-gated attention?": each kept token's score is a bias on the attention
// logits above the gate, scaled by a learnable per-head gain, with a learnable
// temperature).  Per kept query row i and head h:
//   logit_ij = (q'_i . k'_j) / (sqrt(D) tau) + gain_h s_j,  pos_j <= pos_i,
//   o_i = softmax_j(logit_ij) v_j.
//
// Flash-attention forward on tcgen05:
//   * a CTA owns two 128-row query tiles that share one KV head: the two
//     query heads of a GQA pair on the same rows (hq/hkv even), or two
//     consecutive row blocks of one head (hq/hkv odd);
//   * warp 8 streams K and V tiles (128 keys x D) with TMA into a 2-stage
//     ring, plus each key's score and original position;
//   * warp 9 issues the MMAs: S_t = Q_t K^T + (gain_h sqrt(D) tau) s_j into
//     TMEM (fp32, 128 columns per tile), then O_t += P_t V with P_t read
//     straight from TMEM.  The score bias rides in one extra 16-wide K step:
//     Q_t gets the columns (g_hi, g_hi, g_lo) and K the columns (s_hi, s_lo,
//     s_hi), bf16 hi/lo splits of g = gain_h sqrt(D) tau and s_j, so the
//     product carries g s_j to about 2^-16 relative;
//   * warps 0-3 / 4-7 are the softmax warpgroups of tile 0 / tile 1, one
//     thread per query row: they read S from TMEM, fold scale and log2(e)
//     and the causal mask on ORIGINAL positions into the logits, keep the
//     running max/sum (the max only moves when it grows by more than 2^8, so
//     O is rarely rescaled), write P as bf16 back into TMEM over S, and
//     finally normalise O and store it.
//   TMEM: S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [384,384+D).
//
// Keys are visited only up to the query tile's diagonal: positions strictly
// increase inside a sequence (checked by the RoPE prologue), so a key after
// the last query row of the tile has a larger position and is masked anyway.
#include "tg_common.cuh"

namespace tg {

constexpr int kAttnThreads = 384;   // 2 softmax warpgroups + producer/MMA warpgroup
// Register split by setmaxnreg: the kernel launches with kLaunchRegs per
// thread (384 x 168 = 64512); the softmax warpgroups grow to kSoftmaxRegs and
// the producer/MMA warpgroup shrinks to kCtrlRegs, 2*128*192 + 128*112 = 63488.
constexpr int kLaunchRegs = 168;
constexpr int kSoftmaxRegs = 192;
constexpr int kCtrlRegs = 112;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kCtrlRegs <= kAttnThreads * kLaunchRegs, "register split");
constexpr int kTileRows = 128;
constexpr int kKvStages = 2;
constexpr int kMetaSlots = 3;       // key-position slots (one more than the K/V stages)
constexpr float kRescaleThreshold = 8.0f;   // log2 units

// byte offset of row r's first 16-byte core-matrix row in a bias K step
__device__ __forceinline__ uint32_t bias_row_offset(int r) {
  return static_cast<uint32_t>((r >> 3) * 256 + (r & 7) * 16);
}

template <int kD>
struct AttnSmem {
  static constexpr int kTileBytes = kTileRows * kD * 2;   // one 128 x D bf16 tile
  alignas(1024) uint8_t q[2][kTileBytes];
  alignas(1024) uint8_t k[kKvStages][kTileBytes];
  alignas(1024) uint8_t v[kKvStages][kTileBytes];
  // the bias K step, bf16 in no-swizzle K-major core matrices (8 rows x
  // 16 B; the two 8-column halves of a row group 128 B apart, row groups
  // 256 B apart): Q side per tile, K side per stage
  alignas(256) uint8_t qx[2][kTileRows * 32];
  alignas(256) uint8_t kx[kKvStages][kTileRows * 32];
  int32_t kpos[kMetaSlots][kTileRows];
  int32_t kmax[kMetaSlots];
  uint64_t q_full;
  uint64_t k_full[kKvStages];
  uint64_t v_full[kKvStages];
  uint64_t meta_full[kMetaSlots];  // key positions of a tile written
  uint64_t s_full[2][2];            // [tile][step parity]: S_t(j) in TMEM
  uint64_t p_full[2];
  uint64_t o_done[2];              // the last product into O_t done
  uint64_t mma_final[2];
  uint32_t tmem_base;
  volatile int abort;
};

template <int kD>
__global__ void __launch_bounds__(kAttnThreads, 1)
attn_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
            const __grid_constant__ CUtensorMap map_v, AttnArgs a, int n_units_per_rb, int pair_heads) {
  extern __shared__ uint8_t smem_raw[];
  using Smem = AttnSmem<kD>;
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kBoxes = kD / 64;                 // 64-column TMA boxes per tile
  constexpr uint32_t kBoxBytes = kTileRows * 64 * 2;
  constexpr uint32_t kTileBytes = Smem::kTileBytes;

  const int warp = warp_id();
  const int lane = lane_id();
  const int group = a.hq / a.hkv;

  // ---- work unit: longest row blocks first -------------------------------
  const int rb_rev = blockIdx.x / n_units_per_rb;
  const int rest = blockIdx.x - rb_rev * n_units_per_rb;
  const int b = rest % a.batch;
  const int hu = rest / a.batch;
  const int seq_start = __ldg(a.cu_kept + b);
  const int seq_len = __ldg(a.cu_kept + b + 1) - seq_start;
  int head[2], row0[2];
  int n_rb;
  if (pair_heads) {
    n_rb = (a.max_kept + kTileRows - 1) / kTileRows;
    const int rb = n_rb - 1 - rb_rev;
    head[0] = 2 * hu; head[1] = 2 * hu + 1;
    row0[0] = row0[1] = rb * kTileRows;
  } else {
    n_rb = (a.max_kept + 2 * kTileRows - 1) / (2 * kTileRows);
    const int rb = n_rb - 1 - rb_rev;
    head[0] = head[1] = hu;
    row0[0] = rb * 2 * kTileRows;
    row0[1] = row0[0] + kTileRows;
  }
  if (seq_len < 0 || seq_start < 0 || static_cast<long long>(seq_start) + seq_len > a.n_kept) {
    if (threadIdx.x == 0) record_error(a.status, kStatusIndex);
    return;
  }
  if (row0[0] >= seq_len) return;                 // nothing in this sequence
  const int kvh = head[0] / group;
  const int row_end = min(seq_len, row0[1] + kTileRows);
  const int n_kv = (row_end + kTileRows - 1) / kTileRows;

  // ---- setup ---------------------------------------------------------------
  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full, 1);
    for (int s = 0; s < kKvStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.v_full[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.s_full[t][0], 1);
      mbar_init(&sm.s_full[t][1], 1);
      mbar_init(&sm.p_full[t], 128);
      mbar_init(&sm.o_done[t], 1);
    }
    for (int s = 0; s < kMetaSlots; ++s) mbar_init(&sm.meta_full[s], 1);
    mbar_init(&sm.mma_final[0], 1);
    mbar_init(&sm.mma_final[1], 1);
    sm.abort = 0;
    fence_barrier_init();
  }
  if (warp == 9) { tmem_alloc(&sm.tmem_base, 512); tmem_relinquish(); }
  {
    // Q-side bias columns of both tiles; the K side's upper half stays zero
    const int i = threadIdx.x;
    if (i < 2 * kTileRows) {
      const int t = i / kTileRows, r = i % kTileRows;
      const float g = __ldg(a.gain + (t ? head[1] : head[0])) * a.bias_unit;
      const __nv_bfloat16 g_hi = __float2bfloat16_rn(g);
      const __nv_bfloat16 g_lo = __float2bfloat16_rn(g - __bfloat162float(g_hi));
      uint8_t* row = sm.qx[t] + bias_row_offset(r);
      const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(g_hi));
      const uint32_t lo = static_cast<uint32_t>(__bfloat16_as_ushort(g_lo));
      *reinterpret_cast<uint4*>(row) = make_uint4(hi | (hi << 16), lo, 0u, 0u);
      *reinterpret_cast<uint4*>(row + 128) = make_uint4(0u, 0u, 0u, 0u);
    } else {
      const int r = i - 2 * kTileRows;
      for (int s = 0; s < kKvStages; ++s)
        *reinterpret_cast<uint4*>(sm.kx[s] + bias_row_offset(r) + 128) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const long long wd = a.watchdog;
  if (warp >= 8) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
  if (warp == 8) {
    // ======================= producer =======================
    if (lane == 0) {
      prefetch_tmap(&map_q); prefetch_tmap(&map_k); prefetch_tmap(&map_v);
      mbar_arrive_expect_tx(&sm.q_full, 2 * kTileBytes);
      for (int t = 0; t < 2; ++t)
        for (int bx = 0; bx < kBoxes; ++bx)
          tma_load_3d(sm.q[t] + bx * kBoxBytes, &map_q, &sm.q_full, bx * 64, t ? head[1] : head[0],
                      seq_start + (t ? row0[1] : row0[0]));
    }
    // Each key's score (for the bias columns) and position (for the causal
    // mask) are fetched into registers one tile ahead, so that the K/V
    // copies of a freed stage are issued without waiting for those loads.
    float sv[kTileRows / 32];
    int pv[kTileRows / 32];
    auto load_meta = [&](int j) {
#pragma unroll
      for (int u = 0; u < kTileRows / 32; ++u) {
        const int kr = j * kTileRows + u * 32 + lane;
        sv[u] = 0.0f;
        pv[u] = INT_MAX;                          // keys past the sequence end are masked
        if (j < n_kv && kr < seq_len) {
          sv[u] = __ldg(a.s_kept + seq_start + kr);
          pv[u] = __ldg(a.pos + seq_start + kr);
        }
      }
    };
    load_meta(0);
    int issued_k = 0, issued_v = 0;   // tiles whose K / V copies were issued
    int prev_last = -1;               // position of the previous tile's last key
    const bool check_pos = hu == 0 && row_end == seq_len;
    for (int j = 0; j < n_kv; ++j) {
      const int st = j & 1;
      // The MMAs of one thread complete in issue order, so S_1(m) done
      // implies every earlier product done.  K of tile j (and its bias
      // columns) may replace tile j-2's once S_1(j-2) is done; V once
      // PV_1(j-2) is, i.e. once S_1(j-1) is.
      // Each S_1 barrier completes every other step, and the MMAs cannot run
      // two of its phases ahead of this warp (S_1(j) needs the K copy issued
      // here), so a parity wait is unambiguous.
      bool ok = true;
      const int krow = seq_start + j * kTileRows;
      if (lane == 0 && j >= 2) ok = mbar_wait(&sm.s_full[1][st], ((j - 2) >> 1) & 1u, wd, a.status, kStatusTimeout);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok || sm.abort) { sm.abort = 1; break; }
      // K-side bias columns (s_hi, s_lo, s_hi) of this tile's keys; an
      // infinite score keeps (s, 0, 0) so that no 0 * inf appears
#pragma unroll
      for (int u = 0; u < kTileRows / 32; ++u) {
        const float s = sv[u];
        const __nv_bfloat16 s_hi = __float2bfloat16_rn(s);
        const __nv_bfloat16 s_lo = isinf(s) ? __float2bfloat16_rn(0.0f) : __float2bfloat16_rn(s - __bfloat162float(s_hi));
        const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(s_hi));
        const uint32_t lo = static_cast<uint32_t>(__bfloat16_as_ushort(s_lo));
        const uint32_t third = isinf(s) ? 0u : hi;
        *reinterpret_cast<uint4*>(sm.kx[st] + bias_row_offset(u * 32 + lane)) = make_uint4(hi | (lo << 16), third, 0u, 0u);
      }
      // key positions for the softmax, in slot j % 3: the slot's last reader,
      // the softmax of tile j-3, arrived before PV_1(j-3), which precedes
      // S_1(j-2), so the slot is free here, a whole step before the K/V
      // stage is
      {
        const int ms = j % kMetaSlots;
        int kmax = INT_MIN;
#pragma unroll
        for (int u = 0; u < kTileRows / 32; ++u) {
          sm.kpos[ms][u * 32 + lane] = pv[u];
          kmax = max(kmax, pv[u]);
        }
        for (int o = 16; o > 0; o >>= 1) kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
        if (lane == 0) sm.kmax[ms] = kmax;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.meta_full[j % kMetaSlots]);
        mbar_arrive_expect_tx(&sm.k_full[st], kTileBytes);
        for (int bx = 0; bx < kBoxes; ++bx)
          tma_load_3d(sm.k[st] + bx * kBoxBytes, &map_k, &sm.k_full[st], bx * 64, kvh, krow);
        issued_k = j + 1;
        if (j >= 2) ok = mbar_wait(&sm.s_full[1][st ^ 1], ((j - 1) >> 1) & 1u, wd, a.status, kStatusTimeout);
        if (ok) {
          mbar_arrive_expect_tx(&sm.v_full[st], kTileBytes);
          for (int bx = 0; bx < kBoxes; ++bx)
            tma_load_3d(sm.v[st] + bx * kBoxBytes, &map_v, &sm.v_full[st], bx * 64, kvh, krow);
          issued_v = j + 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok || sm.abort) { sm.abort = 1; break; }
      // Positions must be non-negative and strictly increase inside the
      // sequence (the causal tile skipping relies on it).  One CTA per
      // sequence, the first head unit of the row block that reaches the
      // sequence end (it reads every key), checks each key against the next
      // one once its copies are out.
      if (check_pos) {
        bool bad = false;
#pragma unroll
        for (int u = 0; u < kTileRows / 32; ++u) {
          const int kr = j * kTileRows + u * 32 + lane;
          const int down = __shfl_down_sync(0xffffffffu, pv[u], 1);
          const int wrap = __shfl_sync(0xffffffffu, pv[u + 1 < kTileRows / 32 ? u + 1 : u], 0);
          const bool has_next = kr + 1 < seq_len && (lane < 31 || u + 1 < kTileRows / 32);
          const int nxt = lane < 31 ? down : wrap;
          if (kr < seq_len && (pv[u] < 0 || (has_next && nxt <= pv[u]))) bad = true;
        }
        if (lane == 0 && j > 0 && j * kTileRows < seq_len && pv[0] <= prev_last) bad = true;
        if (__any_sync(0xffffffffu, bad) && lane == 0) record_error(a.status, kStatusIndex);
        prev_last = __shfl_sync(0xffffffffu, pv[kTileRows / 32 - 1], 31);
      }
      load_meta(j + 1);
    }
    if (lane == 0) {
      // every issued copy must land before the CTA may leave
      mbar_wait(&sm.q_full, 0, kDrainCycles, a.status, kStatusTimeout);
      auto drain = [&](uint64_t* full, int issued) {
        for (int st = 0; st < kKvStages && st < issued; ++st) {
          const int last = ((issued - 1 - st) / kKvStages) * kKvStages + st;
          mbar_wait(&full[st], static_cast<uint32_t>(last >> 1) & 1u, kDrainCycles, a.status, kStatusTimeout);
        }
      };
      drain(sm.k_full, issued_k);
      drain(sm.v_full, issued_v);
    }
  } else if (warp == 9) {
    // ======================= MMA issuer =======================
    // tcgen05.mma operations of one thread execute in issue order, so
    // S_t(j+1), issued after O_t += P_t(j) V_j, overwrites the TMEM columns
    // of P_t(j) only after that product has read them.  The whole warp runs
    // this loop, so that the descriptors stay warp-uniform, and one elected
    // lane issues; it polls its barriers without suspending (test_wait),
    // which keeps its reaction to a finished softmax short.
    {
      const uint32_t idesc_qk = idesc_bf16_f32(128, 128, 0, 0);
      const uint32_t idesc_pv = idesc_bf16_f32(128, kD, 0, 1);
      // shared-memory descriptors are built once; a K step only advances the
      // start-address field (the low bits, in 16-byte units)
      const uint64_t qd0 = smem_desc_sw128(smem_u32(sm.q[0]), 16, 1024);
      const uint64_t qd1 = smem_desc_sw128(smem_u32(sm.q[1]), 16, 1024);
      const uint64_t kd0 = smem_desc_sw128(smem_u32(sm.k[0]), 16, 1024);
      const uint64_t kd1 = smem_desc_sw128(smem_u32(sm.k[1]), 16, 1024);
      const uint64_t vd0 = smem_desc_sw128(smem_u32(sm.v[0]), kBoxBytes, 1024);
      const uint64_t vd1 = smem_desc_sw128(smem_u32(sm.v[1]), kBoxBytes, 1024);
      const uint64_t qxd0 = smem_desc_interleave(smem_u32(sm.qx[0]), 128, 256);
      const uint64_t qxd1 = smem_desc_interleave(smem_u32(sm.qx[1]), 128, 256);
      const uint64_t kxd0 = smem_desc_interleave(smem_u32(sm.kx[0]), 128, 256);
      const uint64_t kxd1 = smem_desc_interleave(smem_u32(sm.kx[1]), 128, 256);
      auto issue_s = [&](int t, int st, int j) {
        const uint64_t qd = t ? qd1 : qd0;
        const uint64_t kd = st ? kd1 : kd0;
        const uint32_t tS = tmem + static_cast<uint32_t>(t) * 128u;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * kBoxBytes + (ks & 3) * 32) >> 4;
          mma_ss_warp(tS, qd + off, kd + off, idesc_qk, ks > 0 ? 1u : 0u);
        }
        mma_ss_warp(tS, t ? qxd1 : qxd0, st ? kxd1 : kxd0, idesc_qk, 1u);   // + g s_j
        mma_commit_warp(&sm.s_full[t][j & 1]);
      };
      auto issue_pv = [&](int t, int st, int j) {
        const uint64_t vd = st ? vd1 : vd0;
        const uint32_t tS = tmem + static_cast<uint32_t>(t) * 128u;
        const uint32_t tO = tmem + 256u + static_cast<uint32_t>(t) * 128u;
#pragma unroll
        for (int ks = 0; ks < kTileRows / 16; ++ks)
          mma_ts_warp(tO, tS + ks * 8, vd + ((ks * 2048) >> 4), idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
        if (j == n_kv - 1) mma_commit_warp(&sm.o_done[t]);
      };
      // every lane polls; the verdict is made warp-uniform
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait_spin(bar, parity, wd, a.status, kStatusTimeout) && !sm.abort);
      };
      bool ok = wait(&sm.q_full, 0) && wait(&sm.k_full[0], 0);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0, 0);
        issue_s(1, 0, 0);
      }
      for (int j = 0; j < n_kv && ok; ++j) {
        const int st = j & 1;
        const uint32_t use = j >> 1;
        const uint32_t pj = j & 1;
        const bool more = j + 1 < n_kv;
        const int st2 = (j + 1) & 1;
        const uint32_t use2 = (j + 1) >> 1;
        ok = wait(&sm.v_full[st], use & 1u) && wait(&sm.p_full[0], pj);
        if (!ok) break;
        tc_fence_after();
        issue_pv(0, st, j);
        if (more) {
          ok = wait(&sm.k_full[st2], use2 & 1u);
          if (!ok) break;
          issue_s(0, st2, j + 1);
        }
        ok = wait(&sm.p_full[1], pj);
        if (!ok) break;
        tc_fence_after();
        issue_pv(1, st, j);
        if (more) issue_s(1, st2, j + 1);
      }
      if (!ok) sm.abort = 1;
      mma_commit_warp(&sm.mma_final[0]);
      mbar_wait(&sm.mma_final[0], 0, kDrainCycles, a.status, kStatusTimeout);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // ======================= softmax warpgroups =======================
    const int t = warp >> 2;                      // tile
    const int sub = warp & 3;                     // TMEM lane quarter
    const int r = sub * 32 + lane;                // row inside the tile
    const int my_head = t ? head[1] : head[0];
    const int qrow = (t ? row0[1] : row0[0]) + r;
    const bool valid = qrow < seq_len;
    const int qpos = valid ? __ldg(a.pos + seq_start + qrow) : -1;
    const float2 sl = make_float2(a.scale_log2, a.scale_log2);
    const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
    const uint32_t tS = tmem + static_cast<uint32_t>(t * 128) + lane_off;
    const uint32_t tO = tmem + 256u + static_cast<uint32_t>(t * 128) + lane_off;
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int st = j & 1;
      const uint32_t use = j >> 1;
      const int ms = j % kMetaSlots;
      bool w = mbar_wait(&sm.meta_full[ms], static_cast<uint32_t>(j / kMetaSlots) & 1u, wd, a.status, kStatusTimeout);
      w = w && mbar_wait(&sm.s_full[t][st], use & 1u, wd, a.status, kStatusTimeout);
      ok = __all_sync(0xffffffffu, w) && !sm.abort;
      if (!ok) break;
      tc_fence_after();
      // logits in log2 units: x = S * log2(e)/(sqrt(D) tau) (the score bias
      // is already in S), one TMEM read of the whole 128-column row, then
      // max, exp2 and P.
      uint32_t rr[kTileRows];
#pragma unroll
      for (int c = 0; c < kTileRows / 32; ++c)
        tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&rr[c * 32]));
      const bool masked = __any_sync(0xffffffffu, sm.kmax[ms] > qpos);
      const int* kp = sm.kpos[ms];
      tmem_ld_wait();
      // the max is taken on the raw scores (the scale is positive), and the
      // scale and the max meet in one fused multiply-add per pair
      float2 x[kTileRows / 2];
#pragma unroll
      for (int i = 0; i < kTileRows / 2; ++i)
        x[i] = make_float2(__uint_as_float(rr[2 * i]), __uint_as_float(rr[2 * i + 1]));
      if (masked) {
#pragma unroll
        for (int i = 0; i < kTileRows / 2; ++i) {
          if (kp[2 * i] > qpos) x[i].x = -INFINITY;
          if (kp[2 * i + 1] > qpos) x[i].y = -INFINITY;
        }
      }
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < kTileRows / 2; ++i) mx[i & 3] = fmax3(mx[i & 3], x[i].x, x[i].y);
      const float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), mx[3], -INFINITY) * sl.x;
      const float m_new = (mt > m + kRescaleThreshold) ? mt : m;
      const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
      const float alpha = (m_new == m) ? 1.0f : ex2_approx(m - m_use);
      const float2 negm = make_float2(-m_use, -m_use);
      float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int c = 0; c < kTileRows / 32; ++c) {
        uint32_t p16[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 y = __ffma2_rn(x[c * 16 + i], sl, negm);
          const float p0 = ex2_approx(y.x);
          const float p1 = ex2_approx(y.y);
          if (i & 1) acc1 = __fadd2_rn(acc1, make_float2(p0, p1));
          else acc0 = __fadd2_rn(acc0, make_float2(p0, p1));
          p16[i] = pack_bf16x2(p0, p1);
        }
        // P chunk c: bf16 pairs over S columns [16c, 16c + 16)
        tmem_st16(tS + c * 16, p16);
      }
      l = l * alpha + ((acc0.x + acc0.y) + (acc1.x + acc1.y));
      m = m_new;
      // rescale O when this row's max moved (warp-uniform TMEM access); the
      // product into O of step j-1 was issued before S_t(j), so it is done
      if (__any_sync(0xffffffffu, j > 0 && alpha != 1.0f)) {
#pragma unroll
        for (int c = 0; c < kD / 16; ++c) {
          uint32_t o16[16];
          tmem_ld16(tO + c * 16, o16);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) o16[i] = __float_as_uint(__uint_as_float(o16[i]) * alpha);
          tmem_st16(tO + c * 16, o16);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sm.p_full[t]);
    }
    if (!ok) sm.abort = 1;
    // ---- epilogue: O / l -> bf16 ----
    const bool w3 = ok && __all_sync(0xffffffffu,
                                     mbar_wait(&sm.o_done[t], 0, wd, a.status, kStatusTimeout));
    if (w3) {
      tc_fence_after();
      const float inv = 1.0f / l;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.o) +
                            (static_cast<size_t>(seq_start + qrow) * a.hq + my_head) * kD;
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t o32[32];
        tmem_ld32(tO + c * 32, o32);
        tmem_ld_wait();
        if (valid) {
          uint4 v[4];
          uint32_t* pw = reinterpret_cast<uint32_t*>(v);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pw[i] = pack_bf16x2(__uint_as_float(o32[2 * i]) * inv, __uint_as_float(o32[2 * i + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = v[i];
        }
      }
      if (valid && a.lse)
        a.lse[static_cast<size_t>(my_head) * a.n_kept + seq_start + qrow] =
            (((m == -INFINITY) ? 0.0f : m) + __log2f(l)) * 0.6931471805599453f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) { tc_fence_after(); tmem_dealloc(tmem, 512); }
}

template <int kD>
static cudaError_t launch_attn_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                                 const AttnArgs& a, cudaStream_t st) {
  const int group = a.hq / a.hkv;
  const int pair_heads = (group % 2 == 0) ? 1 : 0;
  int n_rb, units_per_rb;
  if (pair_heads) {
    n_rb = (a.max_kept + kTileRows - 1) / kTileRows;
    units_per_rb = a.batch * (a.hq / 2);
  } else {
    n_rb = (a.max_kept + 2 * kTileRows - 1) / (2 * kTileRows);
    units_per_rb = a.batch * a.hq;
  }
  // at least 116 KB so that one CTA (holding all 512 TMEM columns) runs per SM
  size_t smem = sizeof(AttnSmem<kD>) + 1024;
  if (smem < 116 * 1024) smem = 116 * 1024;
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<kD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // the setmaxnreg split is only valid for the launch register count it was
  // sized for; refuse to launch otherwise (setmaxnreg.inc would never return)
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, attn_kernel<kD>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  const long long grid = static_cast<long long>(n_rb) * units_per_rb;
  if (grid == 0) return cudaSuccess;
  attn_kernel<kD><<<static_cast<unsigned>(grid), kAttnThreads, smem, st>>>(mq, mk, mv, a, units_per_rb,
                                                                          pair_heads);
  return cudaGetLastError();
}

cudaError_t launch_attention(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                             const AttnArgs& a, cudaStream_t st) {
  if (a.n_kept == 0 || a.batch == 0) return cudaSuccess;
  if (a.head_dim == 128) return launch_attn_d<128>(mq, mk, mv, a, st);
  return launch_attn_d<64>(mq, mk, mv, a, st);
}

}  // namespace tg
