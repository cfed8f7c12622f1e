// Backward of token-gated attention with respect to the score-side
// parameters: the kept scores s, the per-head gains and the temperature (the
// gradient path from the attention loss back to the gate; TokenGate, "What is
// token-gated attention?": the score enters the logits as gain_h s_j, the
// temperature divides q.k).  For L = sum dO . o, per head h and query row i:
//   P_ij = exp(logit_ij - lse_i),  dP_ij = dO_i . v_j,  D_i = dO_i . o_i,
//   dl_ij = P_ij (dP_ij - D_i)
//   ds_j = sum_h gain_h sum_i dl_ij,   dgain_h = sum_ij s_j dl_ij,
//   dtau = -sum_hij dl_ij (q'_i . k'_j) / (sqrt(D) tau^2).
// dq, dk and dv are not formed.
//
// Kernels:
//   * delta_kernel: D_i = dO_i . o_i per head (one warp per token);
//   * attn_bwd_kernel: CTA pairs (cluster of two, cta_group::2).  A pair owns
//     256 consecutive keys of one KV head, 128 per CTA, and walks the query
//     tiles that can see them (128 rows, from the pair's diagonal to the end of
//     the sequence) for every query head of the group.  Per step the pair's
//     tensor cores compute, TRANSPOSED so that TMEM lanes are keys,
//       S^T  = K Q_h^T   (256 keys x 128 queries, fp32)
//       dP^T = V dO_h^T
//     with each CTA staging its own 128 K/V rows (A) and one half of the
//     step's Q_h / dO_h rows (B, split by the pair).  Every sum over queries
//     then runs along a thread's own TMEM row: one thread per key accumulates
//     sum_i dl_ij and sum_i dl_ij S_ij in registers, with no cross-thread
//     reduction.  Two warpgroups take alternate steps (double-buffered TMEM),
//     so one works while the tensor cores fill the other buffer;
//   * bwd_head_kernel / bwd_ds_kernel: deterministic reductions of the
//     per-key partial sums into dgain, dtau and ds.
#include <climits>

#include "tg_common.cuh"

namespace tg {

constexpr int kBwdThreads = 384;   // warps 0-7: the two warpgroups; 8: copies; 9: MMA; 10: metadata
// Register split by setmaxnreg: launched with kBwdLaunchRegs per thread
// (384 x 168 = 64512), the two warpgroups grow to kBwdSoftRegs and warps
// 8-11 shrink to kBwdCtrlRegs: 2*128*192 + 128*112 = 63488.
constexpr int kBwdLaunchRegs = 168;
constexpr int kBwdSoftRegs = 192;
constexpr int kBwdCtrlRegs = 112;
static_assert(2 * 128 * kBwdSoftRegs + 128 * kBwdCtrlRegs <= kBwdThreads * kBwdLaunchRegs, "register split");
constexpr int kBwdStages = 4;      // Q/dO ring
constexpr int kBwdMeta = 6;        // per-step query metadata slots
constexpr float kLog2e = 1.4426950408889634f;

template <int kD>
struct BwdSmem {
  static constexpr int kKvBytes = 128 * kD * 2;        // this CTA's 128 keys
  static constexpr int kHalfBytes = 64 * kD * 2;       // this CTA's half of a 128-row query tile
  alignas(1024) uint8_t k[kKvBytes];
  alignas(1024) uint8_t v[kKvBytes];
  alignas(1024) uint8_t q[kBwdStages][kHalfBytes];
  alignas(1024) uint8_t dout[kBwdStages][kHalfBytes];
  // per step and query column i: {-L_i, -L_i+1, -D_i, -D_i+1} for column
  // pairs (L = lse log2 e), and the query position (-1: no row)
  alignas(16) float4 ld[kBwdMeta][64];
  int32_t qpos[kBwdMeta][128];
  float gain[kBwdMaxGroup];
  uint64_t kv_full;                  // leader: both CTAs' K and V landed
  uint64_t full[kBwdStages];         // leader: both CTAs' halves of a step landed
  uint64_t ring_free[kBwdStages];    // this CTA's stage may be refilled
  uint64_t meta_full[kBwdMeta];
  uint64_t meta_free[kBwdMeta];
  uint64_t step_full[2];             // S^T and dP^T of a step are in TMEM buffer t
  uint64_t tmem_free[2];             // leader: both CTAs' warpgroups have read buffer t
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t peer_issued;              // leader: stages the other CTA issued
  volatile int abort;
};

// ---------------------------------------------------------------------------
// D_i = dO_i . o_i, written as delta[h * T + i]
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
delta_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ d_o, int64_t n_kept, int hq,
             int head_dim, float* __restrict__ delta) {
  const int lane = lane_id();
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const int vec_per_head = head_dim / 8;            // 16-byte vectors per head: 8 or 16
  const int n_vec = hq * vec_per_head;
  for (long long tok = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + warp_id(); tok < n_kept;
       tok += warps) {
    const uint4* po = reinterpret_cast<const uint4*>(o + tok * hq * head_dim);
    const uint4* pd = reinterpret_cast<const uint4*>(d_o + tok * hq * head_dim);
    for (int v0 = 0; v0 < n_vec; v0 += 32) {
      const int vi = v0 + lane;
      float acc = 0.0f;
      if (vi < n_vec) {
        const uint4 a = __ldg(po + vi);
        const uint4 b = __ldg(pd + vi);
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = __bfloat1622float2(a2[e]);
          const float2 y = __bfloat1622float2(b2[e]);
          acc = fmaf(x.x, y.x, acc);
          acc = fmaf(x.y, y.y, acc);
        }
      }
      // the vec_per_head lanes of one head are consecutive and aligned
      for (int off = vec_per_head >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (vi < n_vec && (lane & (vec_per_head - 1)) == 0) delta[static_cast<long long>(vi / vec_per_head) * n_kept + tok] = acc;
    }
  }
}

// ---------------------------------------------------------------------------
// the pair kernel: per-key partial sums of dl and dl S
// ---------------------------------------------------------------------------
// Work unit (one pair): keys [256 kp, 256 kp + 256) of KV head kvh in sequence
// b; units in order of kp, so the longest ones (kp = 0 sees every query tile)
// start first.  Step n of a unit is query tile qt0 + n / G and query head
// kvh G + n % G; warpgroup t takes the steps n = t mod 2 into TMEM buffer t:
// S^T in columns [256 t, 256 t + 128), dP^T in [256 t + 128, 256 t + 256).
template <int kD>
__global__ void __launch_bounds__(kBwdThreads, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                AttnBwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  using Smem = BwdSmem<kD>;
  // both CTAs of a pair round the same base, so their tiles sit at the same
  // offsets, as the pair MMA's shared-memory descriptors require
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kBoxes = kD / 64;
  constexpr uint32_t kKBox = 128 * 64 * 2;         // 64 columns of 128 keys
  constexpr uint32_t kQBox = 64 * 64 * 2;          // 64 columns of 64 query rows
  constexpr uint32_t kHalf = Smem::kHalfBytes;
  constexpr uint32_t kKv = Smem::kKvBytes;

  const int warp = warp_id();
  const int lane = lane_id();
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int group = a.hq / a.hkv;
  const int unit = static_cast<int>(blockIdx.x >> 1);
  const int per_kp = a.batch * a.hkv;
  const int kp = unit / per_kp;
  const int rest = unit - kp * per_kp;
  const int b = rest % a.batch;
  const int kvh = rest / a.batch;
  const int seq_start = __ldg(a.cu_kept + b);
  const int seq_len = __ldg(a.cu_kept + b + 1) - seq_start;
  if (seq_len < 0 || seq_start < 0 || static_cast<long long>(seq_start) + seq_len > a.n_kept ||
      seq_len > a.max_kept) {
    // a sequence longer than max_kept would leave keys without a unit
    if (threadIdx.x == 0 && leader) record_error(a.status, kStatusIndex);
    return;                                       // both CTAs read the same bounds and leave together
  }
  if (kp * 256 >= seq_len) return;
  const int key0 = kp * 256 + static_cast<int>(rank) * 128;   // this CTA's first key
  const int qt0 = 2 * kp;                         // the first query tile that sees the pair's keys
  const int n_qt = (seq_len + 127) / 128;
  const int n_steps = group * (n_qt - qt0);
  const long long wd = a.watchdog;

  if (threadIdx.x == 0) {
    mbar_init(&sm.kv_full, 1);
    for (int s = 0; s < kBwdStages; ++s) { mbar_init(&sm.full[s], 1); mbar_init(&sm.ring_free[s], 4); }
    for (int s = 0; s < kBwdMeta; ++s) { mbar_init(&sm.meta_full[s], 1); mbar_init(&sm.meta_free[s], 4); }
    for (int t = 0; t < 2; ++t) { mbar_init(&sm.step_full[t], 1); mbar_init(&sm.tmem_free[t], 8); }
    mbar_init(&sm.mma_done, 1);
    sm.abort = 0;
    sm.peer_issued = 0;
    fence_barrier_init();
  }
  if (threadIdx.x < group) sm.gain[threadIdx.x] = __ldg(a.gain + kvh * group + threadIdx.x);
  if (warp == 9) { tmem_alloc_pair(&sm.tmem_base, 512); tmem_relinquish_pair(); }
  tc_fence_before();
  __syncthreads();
  cluster_sync();      // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  uint32_t issued = 0;   // warp 8 lane 0: ring stages this CTA issued
  if (warp >= 8) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kBwdCtrlRegs));
  if (warp == 8) {
    // ======================= copy producer: K/V once, then Q and dO halves =======================
    if (lane == 0) {
      const uint32_t full0 = mapa_shared(smem_u32(&sm.full[0]), 0);
      prefetch_tmap(&map_q); prefetch_tmap(&map_k); prefetch_tmap(&map_v); prefetch_tmap(&map_do);
      const uint32_t kv_bar = mapa_shared(smem_u32(&sm.kv_full), 0);
      if (leader) mbar_arrive_expect_tx(&sm.kv_full, 4 * kKv);
      const int krow = seq_start + key0;
      for (int bx = 0; bx < kBoxes; ++bx) {
        tma_load_2d_pair(sm.k + bx * kKBox, &map_k, kv_bar, kvh * kD + bx * 64, krow);
        tma_load_2d_pair(sm.v + bx * kKBox, &map_v, kv_bar, kvh * kD + bx * 64, krow);
      }
      bool ok = true;
      for (int m = 0; m < n_steps; ++m) {
        const int st = m % kBwdStages;
        if (m >= kBwdStages)
          ok = mbar_wait(&sm.ring_free[st], ((m / kBwdStages) & 1u) ^ 1u, wd, a.status, kStatusTimeout);
        if (!ok || sm.abort) break;
        const int h = kvh * group + m % group;
        const int qrow = seq_start + (qt0 + m / group) * 128 + static_cast<int>(rank) * 64;
        if (leader) mbar_arrive_expect_tx(&sm.full[st], 4 * kHalf);
        for (int bx = 0; bx < kBoxes; ++bx) {
          tma_load_2d_pair(sm.q[st] + bx * kQBox, &map_q, full0 + st * 8u, h * kD + bx * 64, qrow);
          tma_load_2d_pair(sm.dout[st] + bx * kQBox, &map_do, full0 + st * 8u, h * kD + bx * 64, qrow);
        }
        ++issued;
      }
      if (!ok) sm.abort = 1;
      if (!leader) st_cluster_u32(mapa_shared(smem_u32(&sm.peer_issued), 0), issued);
    }
  } else if (warp == 10) {
    // ======================= metadata producer =======================
    // Per step and query column: -lse log2 e (-inf where the row saw no key,
    // so that its P is 0), -D and the position (-1 past the sequence end:
    // masked for every key).  The raw values are loaded kAhead steps ahead
    // into a ring of registers, unconditionally (rows past the sequence read
    // row 0 of it) and with no use until the step is written, so that the L2
    // latency of these loads stays off the step-to-step path.
    constexpr int kAhead = 4;
    float nl[kAhead][4], nd[kAhead][4];
    int qp[kAhead][4];
    auto load_meta = [&](int m, float (&l4)[4], float (&d4)[4], int (&p4)[4]) {
      const int mm = m < n_steps ? m : n_steps - 1;
      const int qt = qt0 + mm / group;
      const int h = kvh * group + mm % group;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        int row = qt * 128 + u * 32 + lane;
        row = row < seq_len ? row : 0;
        const long long gi = static_cast<long long>(h) * a.n_kept + seq_start + row;
        l4[u] = __ldg(a.lse + gi);
        d4[u] = __ldg(a.delta + gi);
        p4[u] = __ldg(a.pos + seq_start + row);
      }
    };
    auto produce = [&](int m, const float (&l4)[4], const float (&d4)[4], const int (&p4)[4]) -> bool {
      const int ms = m % kBwdMeta;
      bool ok = true;
      if (m >= kBwdMeta) {
        if (lane == 0)
          ok = mbar_wait(&sm.meta_free[ms], ((m / kBwdMeta) & 1u) ^ 1u, wd, a.status, kStatusTimeout);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok || sm.abort) return false;
      }
      float* ldf = reinterpret_cast<float*>(sm.ld[ms]);
      const int qt = qt0 + m / group;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = u * 32 + lane;
        const bool in = qt * 128 + c < seq_len;
        const float l = l4[u];
        ldf[(c >> 1) * 4 + (c & 1)] = !in ? 0.0f : (l == -INFINITY ? -INFINITY : -l * kLog2e);
        ldf[(c >> 1) * 4 + 2 + (c & 1)] = in ? -d4[u] : 0.0f;
        sm.qpos[ms][c] = in ? p4[u] : -1;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.meta_full[ms]);
      return true;
    };
#pragma unroll
    for (int r = 0; r < kAhead; ++r) load_meta(r, nl[r], nd[r], qp[r]);
    bool ok = true;
    for (int m0 = 0; m0 < n_steps && ok; m0 += kAhead) {
#pragma unroll
      for (int r = 0; r < kAhead; ++r) {
        const int m = m0 + r;
        if (ok && m < n_steps) {
          ok = produce(m, nl[r], nd[r], qp[r]);
          if (ok) load_meta(m + kAhead, nl[r], nd[r], qp[r]);
        }
      }
    }
    if (!ok) sm.abort = 1;
  } else if (warp == 9) {
    // ======================= pair MMA issuer (leader) =======================
    if (leader && lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(256, 128, 0, 0);
      const uint64_t kd = smem_desc_sw128(smem_u32(sm.k), 16, 1024);
      const uint64_t vd = smem_desc_sw128(smem_u32(sm.v), 16, 1024);
      bool ok = mbar_wait_spin(&sm.kv_full, 0, wd, a.status, kStatusTimeout) && !sm.abort;
      for (int n = 0; n < n_steps && ok; ++n) {
        const int t = n & 1;
        const int st = n % kBwdStages;
        ok = mbar_wait_spin(&sm.full[st], (n / kBwdStages) & 1u, wd, a.status, kStatusTimeout) && !sm.abort;
        // both CTAs' warpgroup t must have read the buffer's previous step
        if (ok && n >= 2)
          ok = mbar_wait_spin(&sm.tmem_free[t], ((n >> 1) & 1u) ^ 1u, wd, a.status, kStatusTimeout) && !sm.abort;
        if (!ok) break;
        tc_fence_after();
        const uint64_t qd = smem_desc_sw128(smem_u32(sm.q[st]), 16, 1024);
        const uint64_t dd = smem_desc_sw128(smem_u32(sm.dout[st]), 16, 1024);
        const uint32_t tS = tmem + static_cast<uint32_t>(t) * 256u;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint32_t ka = ((ks >> 2) * kKBox + (ks & 3) * 32) >> 4;
          const uint32_t qa = ((ks >> 2) * kQBox + (ks & 3) * 32) >> 4;
          mma_ss_pair(tS, kd + ka, qd + qa, idesc, ks > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint32_t ka = ((ks >> 2) * kKBox + (ks & 3) * 32) >> 4;
          const uint32_t qa = ((ks >> 2) * kQBox + (ks & 3) * 32) >> 4;
          mma_ss_pair(tS + 128u, vd + ka, dd + qa, idesc, ks > 0 ? 1u : 0u);
        }
        mma_commit_pair_mc(&sm.step_full[t], 0x3);
      }
      if (!ok) sm.abort = 1;
      // every MMA must have finished before TMEM is freed and either CTA leaves
      mma_commit_pair_mc(&sm.mma_done, 0x1);
      mbar_wait(&sm.mma_done, 0, kDrainCycles, a.status, kStatusTimeout);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kBwdSoftRegs));
    // ======================= the two warpgroups: one thread per key =======================
    const int t = warp >> 2;                      // TMEM buffer / step parity
    const int sub = warp & 3;                     // TMEM lane quarter
    const int krow = key0 + sub * 32 + lane;      // this thread's key (row in the sequence)
    const bool kvalid = krow < seq_len;
    const float sj = kvalid ? __ldg(a.s_kept + seq_start + krow) : 0.0f;
    const int kpos = kvalid ? __ldg(a.pos + seq_start + krow) : INT_MAX;
    const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
    const uint32_t tfree0 = mapa_shared(smem_u32(&sm.tmem_free[0]), 0);
    const float2 c2 = make_float2(a.scale_log2, a.scale_log2);
    float acc_r[kBwdMaxGroup], acc_t[kBwdMaxGroup];
#pragma unroll
    for (int u = 0; u < kBwdMaxGroup; ++u) { acc_r[u] = 0.0f; acc_t[u] = 0.0f; }
    bool ok = true;
    for (int n = t; n < n_steps; n += 2) {
      const int ms = n % kBwdMeta;
      const int st = n % kBwdStages;
      bool w = mbar_wait(&sm.meta_full[ms], static_cast<uint32_t>(n / kBwdMeta) & 1u, wd, a.status, kStatusTimeout);
      w = w && mbar_wait(&sm.step_full[t], static_cast<uint32_t>(n >> 1) & 1u, wd, a.status, kStatusTimeout);
      ok = __all_sync(0xffffffffu, w) && !sm.abort;
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) mbar_arrive(&sm.ring_free[st]);   // the step's MMAs are done with its stage
      const int hh = n % group;
      const int qt = qt0 + n / group;
      // logit in log2 units: S c + gain_h s_j log2 e (-inf for a -inf score)
      const float bj = sm.gain[hh] * sj * kLog2e;
      const float2 b2 = make_float2(bj, bj);
      // only tiles on the diagonal or past the sequence end hold masked entries
      const bool masked = qt * 128 < key0 + 128 || qt * 128 + 128 > seq_len;
      const float4* ld = sm.ld[ms];
      const int* qp = sm.qpos[ms];
      const uint32_t tS = tmem + static_cast<uint32_t>(t) * 256u + lane_off;
      // two 64-column halves: one TMEM wait each, 32 independent column pairs
      float2 r[4], q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) { r[u] = make_float2(0.0f, 0.0f); q[u] = r[u]; }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t rs[64], rp[64];
        tmem_ld32(tS + c * 64, *reinterpret_cast<uint32_t(*)[32]>(&rs[0]));
        tmem_ld32(tS + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&rs[32]));
        tmem_ld32(tS + 128u + c * 64, *reinterpret_cast<uint32_t(*)[32]>(&rp[0]));
        tmem_ld32(tS + 128u + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&rp[32]));
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float4 m4 = ld[c * 32 + i];          // {-L_i, -L_i+1, -D_i, -D_i+1}
          const float2 sv = make_float2(__uint_as_float(rs[2 * i]), __uint_as_float(rs[2 * i + 1]));
          const float2 x = __fadd2_rn(__ffma2_rn(sv, c2, b2), make_float2(m4.x, m4.y));
          float p0 = ex2_approx(x.x);
          float p1 = ex2_approx(x.y);
          if (masked) {
            if (kpos > qp[c * 64 + 2 * i]) p0 = 0.0f;
            if (kpos > qp[c * 64 + 2 * i + 1]) p1 = 0.0f;
          }
          const float2 dp = __fadd2_rn(make_float2(__uint_as_float(rp[2 * i]), __uint_as_float(rp[2 * i + 1])),
                                       make_float2(m4.z, m4.w));
          const float2 dl = __fmul2_rn(make_float2(p0, p1), dp);
          r[i & 3] = __fadd2_rn(r[i & 3], dl);
          q[i & 3] = __ffma2_rn(dl, sv, q[i & 3]);
        }
      }
      // this warp is done with the TMEM buffer and the metadata slot
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_cluster_relaxed(tfree0 + static_cast<uint32_t>(t) * 8u);
        mbar_arrive(&sm.meta_free[ms]);
      }
      const float step_r = ((r[0].x + r[0].y) + (r[1].x + r[1].y)) + ((r[2].x + r[2].y) + (r[3].x + r[3].y));
      const float step_t = ((q[0].x + q[0].y) + (q[1].x + q[1].y)) + ((q[2].x + q[2].y) + (q[3].x + q[3].y));
#pragma unroll
      for (int u = 0; u < kBwdMaxGroup; ++u)
        if (u == hh) { acc_r[u] += step_r; acc_t[u] += step_t; }
    }
    if (!ok) sm.abort = 1;
    if (ok && kvalid) {
#pragma unroll
      for (int u = 0; u < kBwdMaxGroup; ++u) {
        if (u < group) {
          const long long gi = static_cast<long long>(t * a.hq + kvh * group + u) * a.n_kept + seq_start + krow;
          a.r_part[gi] = acc_r[u];
          a.t_part[gi] = acc_t[u];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();      // every role is done; the other CTA's issue count is in place
  if (leader && warp == 8 && lane == 0) {
    // Every copy either CTA issued must land before the pair may leave.  The
    // producers stop together unless a wait ran out; then the leader settles
    // the difference on its stage barriers: it arrives for a stage only the
    // other CTA issued, and counts off the other CTA's half of a stage it
    // issued alone.
    const uint32_t peer = sm.peer_issued;
    for (uint32_t g = issued; g < peer; ++g) mbar_arrive_expect_tx(&sm.full[g % kBwdStages], 2 * kHalf);
    for (uint32_t g = peer; g < issued; ++g) mbar_complete_tx(&sm.full[g % kBwdStages], 2 * kHalf);
    const uint32_t last_g = issued > peer ? issued : peer;
    for (uint32_t st = 0; st < static_cast<uint32_t>(kBwdStages) && st < last_g; ++st) {
      const uint32_t last = ((last_g - 1 - st) / kBwdStages) * kBwdStages + st;
      mbar_wait(&sm.full[st], (last / kBwdStages) & 1u, kDrainCycles, a.status, kStatusTimeout);
    }
    mbar_wait(&sm.kv_full, 0, kDrainCycles, a.status, kStatusTimeout);
  }
  __syncthreads();
  cluster_sync();      // no CTA leaves while the other may still signal it
  if (warp == 9) { tc_fence_after(); tmem_dealloc_pair(tmem, 512); }
}

// ---------------------------------------------------------------------------
// reductions, in a fixed order (bit-reproducible results):
//   bwd_head_kernel, block (c, h): partial sums over key chunk c of
//     sum_j s_j R_hj and sum_j T_hj into part[h][c] (R, T: the two
//     warpgroups' partial sums added; keys past cu_kept[batch] hold none);
//   bwd_ds_kernel: ds_j = sum_h gain_h R_hj per key; block 0 also forms
//     dgain_h = sum_c part_g[h][c] and dtau = dtau_scale sum_h sum_c part_t[h][c].
// ---------------------------------------------------------------------------
__device__ __forceinline__ float block_sum_256(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane_id() == 0) red[warp_id()] = v;
  __syncthreads();
  float s = 0.0f;
  if (threadIdx.x == 0)
    for (int w = 0; w < 8; ++w) s += red[w];
  __syncthreads();
  return s;
}

__global__ void __launch_bounds__(256) bwd_head_kernel(AttnBwdArgs a) {
  __shared__ float red[8];
  const int c = blockIdx.x;
  const int h = blockIdx.y;
  const long long n = a.n_kept;
  const long long n_rows = min(max(static_cast<long long>(__ldg(a.cu_kept + a.batch)), 0LL), n);
  const long long chunk = (n_rows + kBwdChunks - 1) / kBwdChunks;
  const long long j0 = c * chunk;
  const long long j1 = min(n_rows, j0 + chunk);
  const float* r0 = a.r_part + static_cast<long long>(h) * n;
  const float* r1 = a.r_part + static_cast<long long>(a.hq + h) * n;
  const float* t0 = a.t_part + static_cast<long long>(h) * n;
  const float* t1 = a.t_part + static_cast<long long>(a.hq + h) * n;
  float g = 0.0f, tt = 0.0f;
  for (long long j = j0 + threadIdx.x; j < j1; j += 256) {
    const float r = r0[j] + r1[j];
    const float s = __ldg(a.s_kept + j);
    if (r != 0.0f && isfinite(s)) g = fmaf(s, r, g);
    tt += t0[j] + t1[j];
  }
  g = block_sum_256(g, red);
  tt = block_sum_256(tt, red);
  if (threadIdx.x == 0) {
    a.part[(static_cast<long long>(h) * kBwdChunks + c) * 2] = g;
    a.part[(static_cast<long long>(h) * kBwdChunks + c) * 2 + 1] = tt;
  }
}

__global__ void __launch_bounds__(256) bwd_ds_kernel(AttnBwdArgs a) {
  __shared__ float tsum[256];
  const long long j = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
  const long long n = a.n_kept;
  const long long n_rows = min(max(static_cast<long long>(__ldg(a.cu_kept + a.batch)), 0LL), n);
  if (j < n) {
    float acc = 0.0f;
    if (j < n_rows)
      for (int h = 0; h < a.hq; ++h)
        acc = fmaf(__ldg(a.gain + h), a.r_part[static_cast<long long>(h) * n + j] +
                                          a.r_part[static_cast<long long>(a.hq + h) * n + j], acc);
    a.ds[j] = acc;
  }
  if (blockIdx.x == 0) {
    // one thread per head (the host checks hq <= kBwdMaxHeads = 256), then thread 0 over heads
    for (int h = threadIdx.x; h < a.hq; h += 256) {
      float g = 0.0f, tt = 0.0f;
      for (int c = 0; c < kBwdChunks; ++c) {
        g += a.part[(static_cast<long long>(h) * kBwdChunks + c) * 2];
        tt += a.part[(static_cast<long long>(h) * kBwdChunks + c) * 2 + 1];
      }
      a.dgain[h] = g;
      if (h < 256) tsum[h] = tt;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float tt = 0.0f;
      for (int h = 0; h < a.hq && h < 256; ++h) tt += tsum[h];
      *a.dtau = tt * a.dtau_scale;
    }
  }
}

template <int kD>
static cudaError_t launch_bwd_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                                const CUtensorMap& mdo, const AttnBwdArgs& a, cudaStream_t st) {
  // at least 116 KB, so that one CTA (holding all 512 TMEM columns) runs per
  // SM: two pairs sharing two SMs could otherwise each hold one SM's TMEM
  // while waiting for the other's
  size_t smem = sizeof(BwdSmem<kD>) + 1024;
  if (smem < 116 * 1024) smem = 116 * 1024;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<kD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // the setmaxnreg split is only valid for the launch register count it was
  // sized for; refuse to launch otherwise (setmaxnreg.inc would never return)
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, attn_bwd_kernel<kD>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kBwdLaunchRegs) return cudaErrorInvalidConfiguration;
  const long long n_kp = (static_cast<long long>(a.max_kept) + 255) / 256;
  const long long units = n_kp * a.batch * a.hkv;
  if (units == 0) return cudaSuccess;
  if (2 * units > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * units));
  cfg.blockDim = dim3(kBwdThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_bwd_kernel<kD>, mq, mk, mv, mdo, a);
}

cudaError_t launch_attention_bwd(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                                 const CUtensorMap& mdo, const AttnBwdArgs& a, cudaStream_t st) {
  if (a.n_kept == 0 || a.batch == 0) return cudaSuccess;
  {
    const long long warps_needed = a.n_kept;
    long long blocks = (warps_needed + 7) / 8;
    const long long cap = static_cast<long long>(a.num_sms) * 8;
    if (blocks > cap) blocks = cap;
    delta_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(a.o),
                                                               static_cast<const __nv_bfloat16*>(a.d_o), a.n_kept,
                                                               a.hq, a.head_dim, a.delta);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = (a.head_dim == 128) ? launch_bwd_d<128>(mq, mk, mv, mdo, a, st)
                                      : launch_bwd_d<64>(mq, mk, mv, mdo, a, st);
  if (e != cudaSuccess) return e;
  bwd_head_kernel<<<dim3(kBwdChunks, a.hq), 256, 0, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_ds_kernel<<<static_cast<unsigned>((a.n_kept + 255) / 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace tg
