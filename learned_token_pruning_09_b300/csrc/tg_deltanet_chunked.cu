// Pruned Gated DeltaNet scan in chunked form on the tensor cores (TokenGate
// prunes the Gated DeltaNet layers of the hybrid Qwen3.5 model: MarkTechPost
// article, "Does it work on hybrid attention models?"; the recurrence is the
// gated delta rule of Gated DeltaNet, Yang, Kautz and Hatamizadeh).
//
// Per sequence and value head the kept tokens are cut into chunks of 64.
// Within a chunk with entering state S0 [dv, dk], cumulative log-decays
// G_i = sum_{j<=i} g_j, gamma_i = exp(G_i), gamma_C = gamma of the last token:
//   A_ij = beta_i exp(G_i - G_j) k^_i.k^_j  (j < i),   T = (I + A)^-1
//   W1 = T (beta v),  W2 = T (beta gamma k^)
//   Mq_ij = exp(G_i - G_j) q^_i.k^_j  (j <= i)
//   U  = W1 - W2 S0^T                              (the chunk's pseudo-values)
//   O  = (gamma q^ - Mq W2) S0^T + Mq W1 = Qe S0^T + Oloc
//   S  = gamma_C S0 + U^T (exp(G_C - G) k^)
// which is the recurrence token by token, regrouped (the WY form).
//
// Two parts:
//   the per-chunk products, one unit per (chunk, value head), all in
//     parallel: Gram products [k^; q^] k^^T (tf32 MMA), T by forward
//     substitution, W1^T, W2^T (tf32 MMA), Qe, Oloc^T (tf32 MMA); written to
//     the workspace, the state carry's MMA operands as ready shared-memory
//     images (128-byte swizzle, K-major);
//   the state carry, one CTA per (sequence, value head): the state S lives
//     in tensor memory (lane = value row, column = key dim) and is the A
//     operand of both MMAs of a chunk:
//       D = S [W2; Qe]^T          (U = W1 - D1 and O = D3 + Oloc)
//       S = gamma_C S + U^T Kd    (U^T back in tensor memory as the A operand)
//     with the next chunk's operands copied in by the bulk-copy engine while
//     the current one runs.
// With few (sequence, head) pairs both run in one cooperative launch
// (delta_fused_kernel: the carries on some SMs, units on the others, handed
// over by flags); otherwise as two launches (delta_prep_kernel, one CTA per
// unit, then delta_chain_kernel).  The arithmetic is the same either way.
// tf32 MMAs on fp32 operands rounded to nearest (cvt.rna) where they are
// written; fp32 accumulation, fp32 state; o rounded once to bf16.
#include <algorithm>

#include "tg_common.cuh"

namespace tg {

constexpr int kChunk = 64;
constexpr int kAStride = 68;          // row stride (floats) of the plain A matrix: 16-byte rows, 4-way stores
constexpr int kPrepThreads = 128;

__device__ __forceinline__ float to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// Instruction descriptor, kind::tf32: A and B tf32, fp32 accumulation, both
// operands K-major.
__host__ __device__ constexpr uint32_t idesc_tf32_f32(uint32_t m, uint32_t n) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32_ss_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
__device__ __forceinline__ void mma_tf32_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void bulk_copy_g2s(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst_smem)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void bulk_copy_s2g(void* dst, const void* src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               ::"l"(dst), "r"(smem_u32(src_smem)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Byte offset of fp32 element (r, k) in a K-major tile with 128-byte swizzle:
// K-blocks of 32 elements, each `rows` rows of 128 bytes; the 16-byte chunk
// c of row r sits at chunk c ^ (r mod 8).  The tile base is 1024-aligned.
__host__ __device__ __forceinline__ uint32_t sw_off(int rows, int r, int k) {
  return static_cast<uint32_t>((k >> 5) * rows * 128 + r * 128 + ((((k >> 2) & 7) ^ (r & 7)) << 4) + ((k & 3) << 2));
}
// Descriptor start offset (bytes) of K step ks (8 tf32 elements) of such a tile.
__host__ __device__ __forceinline__ uint32_t sw_kstep(int rows, int ks) {
  return static_cast<uint32_t>((ks >> 2) * rows * 128 + (ks & 3) * 32);
}

// Cross-CTA hand-off of a finished unit within one (cooperative) launch: the
// writer group's stores, a barrier of the group, then one release store of
// the unit's flag; readers poll the flag with acquire loads, a bounded wait.
// The state carry reads part of the unit with the bulk-copy engine, so both
// sides also fence the generic stores for the async proxy.
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ bool flag_wait(const int* f, long long limit, unsigned int* status) {
  if (ld_acquire_gpu(f) != 0) return true;
  const long long t0 = clock64();
  while (true) {
    __nanosleep(32);
    if (ld_acquire_gpu(f) != 0) return true;
    if (clock64() - t0 > limit) {
      record_error(status, kStatusTimeout);
      return false;
    }
  }
}

// The workspace, per (chunk slot x, value head h), unit u = x * hv + h:
//   bq  [u][128 rows][dk]  W2 (rows 0..63) and Qe (rows 64..127), swizzled image
//   kd  [u][dk rows][64]   Kd^T = (exp(G_C - G_t) k^_t)^T, swizzled image
//   w1  [u][64][dv]        W1 (token rows), plain fp32
//   ol  [u][64][dv]        Oloc (token rows), plain fp32
//   gc  [u]                gamma_C
//   flag [u]               int, set once unit u is complete (one-launch form only),
//                          then a 64-bit count of the units handed out
// (gc, the flags and the counter fit the 16 bytes per unit added to the size)
// Chunk c of sequence b takes slot floor(cu[b] / 64) + b + c: distinct for
// distinct (b, c), below n_kept / 64 + batch + 1.
struct ChunkWs {
  float* bq;
  float* kd;
  float* w1;
  float* ol;
  float* gc;
  int* flag;
};
__host__ __device__ inline long long chunk_slots(long long n_kept, int batch) { return n_kept / kChunk + batch + 1; }
__host__ __device__ inline ChunkWs chunk_ws(void* base, long long slots, int hv, int dk, int dv) {
  const long long units = slots * hv;
  ChunkWs w;
  char* p = static_cast<char*>(base);
  w.bq = reinterpret_cast<float*>(p);
  p += units * 128LL * dk * 4;
  w.kd = reinterpret_cast<float*>(p);
  p += units * static_cast<long long>(dk) * kChunk * 4;
  w.w1 = reinterpret_cast<float*>(p);
  p += units * static_cast<long long>(dv) * kChunk * 4;
  w.ol = reinterpret_cast<float*>(p);
  p += units * static_cast<long long>(dv) * kChunk * 4;
  w.gc = reinterpret_cast<float*>(p);
  p += units * 4;
  w.flag = reinterpret_cast<int*>(p);
  return w;
}
size_t delta_chunked_ws_bytes(long long n_kept, int batch, int hv, int dk, int dv) {
  const long long units = chunk_slots(n_kept, batch) * hv;
  return static_cast<size_t>(units) * (128ull * dk * 4 + static_cast<size_t>(dk) * kChunk * 4 +
                                       2ull * dv * kChunk * 4 + 16);
}

// ---------------------------------------------------------------------------
// per-chunk products
// ---------------------------------------------------------------------------
// A unit is written for a small instruction footprint (rolled loops over
// 16-byte pieces and 16-column TMEM tiles, rows re-read from L1/L2 rather than
// held in registers) and a small shared-memory and TMEM share, so that three
// units (three CTAs, or three groups of one CTA) fit an SM and hide one
// another's latencies: every MMA operand passes
// through one 32 KB buffer (the Gram product in 64-wide halves of the key
// dims, then the four other products one after another), and the
// accumulators use 128 TMEM columns.
template <int DK>
struct PrepSmem {
  alignas(1024) uint8_t buf[2 * 128 * 128];        // one [128 rows][64] fp32 MMA A operand (2 K-blocks)
  alignas(1024) uint8_t at[kChunk * kAStride * 4];   // A (plain rows), then T (swizzled [i][j])
  alignas(1024) uint8_t mq[kChunk * kChunk * 4];   // Mq, swizzled [i][j]
  float G[kChunk];
  float beta[kChunk];
  float gam[kChunk];                        // exp(G)
  float rn[128];                            // 1 / |k_t| (rows 0..63), scale / |q_t| (64..127)
  uint64_t bar;
  uint32_t tmem_base;
  long long next_unit;                      // one-launch form: the group's next unit, from its thread 0
};

// 8 bf16 (one 16-byte piece) to fp32
__device__ __forceinline__ void bf16x8(const uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}

// One (chunk slot x, value head h) unit of the per-chunk products, by a group
// of 128 threads (tid 0..127, four whole warps aligned to a multiple of four)
// that owns `sm`, the TMEM columns tmem .. tmem + 127, the mbarrier sm.bar
// (its phase count in `phase`, carried from unit to unit) and the named
// barrier bar_id (the group).  A slot that holds no chunk returns at once (the
// same for the whole group).
template <int DK>
__device__ __forceinline__ void delta_prep_unit(const ScanArgs& a, long long slots, int x, int h, PrepSmem<DK>& sm,
                                             int tid, uint32_t tmem, uint32_t& phase, bool& ok, int bar_id) {
  const int warp = tid >> 5, lane = tid & 31;
  auto gbar = [&]() { asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory"); };
  // the sequence of this slot: the largest b with floor(cu[b] / 64) + b <= x
  int lo = 0, hi = a.batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.cu_kept + mid) / kChunk + mid <= x) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int t_seq0 = __ldg(a.cu_kept + b), t_seq1 = __ldg(a.cu_kept + b + 1);
  const int c = x - (t_seq0 / kChunk + b);
  const int len = t_seq1 - t_seq0;
  // a slot no chunk uses, or a sequence outside the tokens (the state-carry
  // kernel flags it)
  if (t_seq0 < 0 || static_cast<long long>(t_seq1) > a.n_kept) return;
  if (c < 0 || len <= 0 || c * kChunk >= len) return;
  const int t0 = t_seq0 + c * kChunk;
  const int n = min(kChunk, len - c * kChunk);
  const int dv = a.dv;
  const int kh = h / (a.hv / a.hk);
  const ChunkWs ws = chunk_ws(a.ws, slots, a.hv, DK, dv);
  const long long u = static_cast<long long>(x) * a.hv + h;
  float* bq = ws.bq + u * 128 * DK;
  float* kdT = ws.kd + u * DK * kChunk;
  const uint32_t bufa = smem_u32(sm.buf), at = smem_u32(sm.at), mq = smem_u32(sm.mq);
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  // After a wait that runs out the same phase is waited for again with the
  // drain limit, so that every MMA has completed before its operands are
  // rewritten and the phases stay in step (the results are then flagged by
  // the status word, not used).
  auto mma_wait = [&]() {
    if (!mbar_wait(&sm.bar, phase & 1u, ok ? a.watchdog : kDrainCycles, a.status, kStatusTimeout)) {
      ok = false;
      mbar_wait(&sm.bar, phase & 1u, kDrainCycles, a.status, kStatusTimeout);
    }
    ++phase;
    tc_fence_after();
  };
  // one MMA of M 128, N 64 over K = 64 (8 steps) from the buffer and a B tile
  // whose K-blocks hold b_rows rows (64 for T and Mq, 128 for the buffer itself)
  auto mma_buf = [&](uint32_t d_col, uint32_t b_addr, int b_rows, bool accumulate) {
    if (warp == 0) {
      tc_fence_after();
      const uint32_t idesc = idesc_tf32_f32(128, 64);
      const uint64_t da = smem_desc_sw128(bufa, 16, 1024);
      const uint64_t db = smem_desc_sw128(b_addr, 16, 1024);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_tf32_ss_warp(tmem + d_col, da + (sw_kstep(128, ks) >> 4), db + (sw_kstep(b_rows, ks) >> 4),
                         idesc, (accumulate || ks > 0) ? 1u : 0u);
      mma_commit_warp(&sm.bar);
    }
  };
  auto to_async = [&]() {                   // this thread's shared-memory writes, then the group
    fence_proxy_async_smem();
    tc_fence_before();
    gbar();
  };

  // 0. cumulative log-decays and write strengths of the chunk
  if (warp == 0) {
    float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
    if (lane < n) { g0 = __ldg(a.g + static_cast<long long>(t0 + lane) * a.hv + h); b0 = __ldg(a.beta + static_cast<long long>(t0 + lane) * a.hv + h); }
    if (lane + 32 < n) { g1 = __ldg(a.g + static_cast<long long>(t0 + lane + 32) * a.hv + h); b1 = __ldg(a.beta + static_cast<long long>(t0 + lane + 32) * a.hv + h); }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v0 = __shfl_up_sync(0xffffffffu, g0, o), v1 = __shfl_up_sync(0xffffffffu, g1, o);
      if (lane >= o) { g0 += v0; g1 += v1; }
    }
    g1 += __shfl_sync(0xffffffffu, g0, 31);
    sm.G[lane] = g0; sm.G[lane + 32] = g1;
    sm.gam[lane] = expf(g0); sm.gam[lane + 32] = expf(g1);
    sm.beta[lane] = b0; sm.beta[lane + 32] = b1;
  }
  tc_fence_before();
  gbar();
  tc_fence_after();
  const float GC = sm.G[kChunk - 1];      // padded tokens have g = 0
  const int t = tid & 63;
  const bool is_k = tid < kChunk;
  const bool valid_t = t < n;
  const uint4* krow = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.k) +
                                                     (static_cast<long long>(t0 + t) * a.hk + kh) * DK);
  const uint4* src = is_k ? krow : reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) +
                                                                  (static_cast<long long>(t0 + t) * a.hk + kh) * DK);
  const int row = is_k ? t : 64 + t;

  // 1. the norms of the k (threads 0..63) and q (64..127) rows; the q threads
  //    also start their token's v row (read in step 5) on its way into L2
  if (!is_k && valid_t) {
    const char* vr = reinterpret_cast<const char*>(static_cast<const uint16_t*>(a.v) +
                                                   (static_cast<long long>(t0 + t) * a.hv + h) * dv);
    asm volatile("prefetch.global.L2 [%0];" ::"l"(vr));              // a row is at most 256 bytes
    if (dv > 64) asm volatile("prefetch.global.L2 [%0];" ::"l"(vr + 128));
  }
  {
    float ss = 0.f;
#pragma unroll 4
    for (int p = 0; p < DK / 8; ++p) {
      float f[8];
      bf16x8(valid_t ? __ldg(src + p) : make_uint4(0, 0, 0, 0), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
    }
    sm.rn[row] = (is_k ? 1.f : a.scale) * rsqrtf(ss + 1e-6f);
  }
  // 2. D[0..63] = [k^; q^] k^^T over the key dims in halves of 64: each half
  //    of the rows into the buffer (tf32), with Kd^T and gamma q^ of those dims
  //    to the workspace, then its MMA
  for (int hf = 0; hf < DK / 64; ++hf) {
    if (hf > 0) gbar();                     // every thread has read the previous half
    const float rn = sm.rn[row];
    const float kdc = expf(GC - sm.G[t]);
#pragma unroll 2
    for (int p = 0; p < 8; ++p) {
      float f[8];
      bf16x8(valid_t ? __ldg(src + hf * 8 + p) : make_uint4(0, 0, 0, 0), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] *= rn;
      *reinterpret_cast<float4*>(sm.buf + sw_off(128, row, 8 * p)) =
          make_float4(to_tf32(f[0]), to_tf32(f[1]), to_tf32(f[2]), to_tf32(f[3]));
      *reinterpret_cast<float4*>(sm.buf + sw_off(128, row, 8 * p + 4)) =
          make_float4(to_tf32(f[4]), to_tf32(f[5]), to_tf32(f[6]), to_tf32(f[7]));
      if (is_k) {
        // Kd^T image: rows (key dims) 64 hf + 8p .. +7, column t (token)
#pragma unroll
        for (int e = 0; e < 8; ++e) kdT[sw_off(DK, hf * 64 + 8 * p + e, t) >> 2] = to_tf32(kdc * f[e]);
      }
    }
    to_async();
    // gamma q^ into the bq image rows 64..127 (completed to Qe in step 8): the
    // buffer's q^ rows have the image's layout (K-blocks of 32 dims, 128 rows),
    // so whole 16-byte pieces go out, consecutive threads on consecutive pieces
    for (int e = tid; e < 2 * 512; e += kPrepThreads) {
      const int kb = e >> 9, rr = (e >> 3) & 63;
      const uint32_t off = kb * 16384 + (64 + rr) * 128 + (e & 7) * 16;
      float4 v = *reinterpret_cast<const float4*>(sm.buf + off);
      const float gm = sm.gam[rr];
      v.x *= gm; v.y *= gm; v.z *= gm; v.w *= gm;
      *reinterpret_cast<float4*>(reinterpret_cast<char*>(bq) + (2 * hf + kb) * 16384 + (64 + rr) * 128 + (e & 7) * 16) = v;
    }
    mma_buf(0, bufa, 128, hf > 0);          // B: the buffer's k^ rows 0..63
    mma_wait();
  }
  // 3. A (plain rows, threads 0..63) and Mq (swizzled, 64..127) from the Gram
  //    products; exp(G_i - G_j) <= 1 for j <= i on the ex2 unit (relative
  //    error ~2^-22)
  {
    const int i = t;
    const float Gi = sm.G[i] * 1.44269504088896341f;
    float* arow = reinterpret_cast<float*>(sm.at) + i * kAStride;
    const float bi = sm.beta[i];
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      uint32_t r[16];
      tmem_ld16(tmem + lane_base + q * 16, r);
      tmem_ld_wait();
#pragma unroll
      for (int j4 = 0; j4 < 16; j4 += 4) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = q * 16 + j4 + e;
          const float ex = ex2_approx(fminf(Gi - sm.G[j] * 1.44269504088896341f, 0.f));
          const float gv = __uint_as_float(r[j4 + e]);
          v[e] = is_k ? ((j < i) ? bi * ex * gv : 0.f) : ((j <= i) ? to_tf32(ex * gv) : 0.f);
        }
        const int j = q * 16 + j4;
        if (is_k)
          *reinterpret_cast<float4*>(arow + j) = make_float4(v[0], v[1], v[2], v[3]);
        else
          *reinterpret_cast<float4*>(sm.mq + sw_off(kChunk, i, j)) = make_float4(v[0], v[1], v[2], v[3]);
      }
    }
  }
  tc_fence_before();
  gbar();
  // this thread's half of its token's v row (read again in step 5), loaded
  // now so that the loads overlap the T solve
  const uint4* vrow = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.v) +
                                                     (static_cast<long long>(t0 + t) * a.hv + h) * dv);
  const int vp0 = is_k ? 0 : dv / 16;
  uint4 vpiece[8];                          // dv / 16 <= 8 pieces
#pragma unroll
  for (int i = 0; i < 8; ++i)
    vpiece[i] = (i < dv / 16 && valid_t) ? __ldg(vrow + vp0 + i) : make_uint4(0, 0, 0, 0);
  // 4. T = (I + A)^-1 in 2 x 2 blocks of 32 (A strictly lower triangular):
  //    the diagonal blocks T11 = (I + A11)^-1 and T22 = (I + A22)^-1 by
  //    forward substitution, T_i = e_i - sum_{j<i} A_ij T_j (warps 0 and 1 at
  //    the same time, one column per lane, in registers); then Y = T22 A21
  //    (warps 1 and 3, 16 rows each) and T21 = -Y T11 (warps 0 and 2); T12 = 0.
  //    The scratch for T11, T22 and Y is the (free) buffer.
  {
    float (*t11)[36] = reinterpret_cast<float(*)[36]>(sm.buf);
    float (*tsc)[36] = reinterpret_cast<float(*)[36]>(sm.buf + 32 * 36 * 4);
    float (*ysc)[36] = reinterpret_cast<float(*)[36]>(sm.buf + 2 * 32 * 36 * 4);
    const int k = lane;
    const float* A = reinterpret_cast<const float*>(sm.at);
    if (warp < 2) {
      const int o = warp * 32;             // the block's first row and column
      float tc[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) tc[i] = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float s0 = (i == k) ? 1.f : 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
        for (int j4 = 0; j4 < (i + 3) / 4; ++j4) {
          const float4 av = *reinterpret_cast<const float4*>(A + (o + i) * kAStride + o + 4 * j4);
          s0 = fmaf(-av.x, tc[4 * j4], s0);
          s1 = fmaf(-av.y, tc[4 * j4 + 1], s1);
          s2 = fmaf(-av.z, tc[4 * j4 + 2], s2);
          s3 = fmaf(-av.w, tc[4 * j4 + 3], s3);
        }
        tc[i] = (s0 + s1) + (s2 + s3);
      }
      float (*dst)[36] = warp == 0 ? t11 : tsc;   // [row][column]
#pragma unroll
      for (int i = 0; i < 32; ++i) dst[i][k] = tc[i];
    }
    gbar();                                 // T11 and T22 in the scratch
    const int i0 = (warp >> 1) * 16;        // this warp's 16 rows of Y or T21
    if (warp & 1) {
      // Y = T22 A21, column k: A21's column in registers, T22's rows broadcast
      float ac[32];
#pragma unroll
      for (int m = 0; m < 32; ++m) ac[m] = A[(32 + m) * kAStride + k];
#pragma unroll 1
      for (int i = i0; i < i0 + 16; ++i) {
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
        for (int m4 = 0; m4 < 8; ++m4) {
          const float4 tv = *reinterpret_cast<const float4*>(&tsc[i][4 * m4]);
          s0 = fmaf(tv.x, ac[4 * m4], s0);
          s1 = fmaf(tv.y, ac[4 * m4 + 1], s1);
          s2 = fmaf(tv.z, ac[4 * m4 + 2], s2);
          s3 = fmaf(tv.w, ac[4 * m4 + 3], s3);
        }
        ysc[i][k] = (s0 + s1) + (s2 + s3);
      }
    }
    gbar();                                 // Y complete; A is read, so T may overwrite it
    if (!(warp & 1)) {
      // T21 = -Y T11 (column k of T11 in registers), and T11's rows i0..i0+15
      float tk[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) tk[j] = t11[j][k];
#pragma unroll 1
      for (int i = i0; i < i0 + 16; ++i) {
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 yv = *reinterpret_cast<const float4*>(&ysc[i][4 * j4]);
          s0 = fmaf(-yv.x, tk[4 * j4], s0);
          s1 = fmaf(-yv.y, tk[4 * j4 + 1], s1);
          s2 = fmaf(-yv.z, tk[4 * j4 + 2], s2);
          s3 = fmaf(-yv.w, tk[4 * j4 + 3], s3);
        }
        *reinterpret_cast<float*>(sm.at + sw_off(kChunk, 32 + i, k)) = to_tf32((s0 + s1) + (s2 + s3));
        *reinterpret_cast<float*>(sm.at + sw_off(kChunk, i, k)) = to_tf32(t11[i][k]);
      }
    } else {
      // T22's rows i0..i0+15, and T12 = 0
#pragma unroll 1
      for (int i = i0; i < i0 + 16; ++i) {
        *reinterpret_cast<float*>(sm.at + sw_off(kChunk, 32 + i, 32 + k)) = to_tf32(tsc[i][k]);
        *reinterpret_cast<float*>(sm.at + sw_off(kChunk, i, 32 + k)) = 0.f;
      }
    }
  }
  tc_fence_before();
  gbar();
  // 5. W1^T = (beta v)^T T^T (TMEM 64..127), then W2^T = (beta gamma k^)^T T^T
  //    (TMEM 0..63), each right-hand side through the buffer, column t from
  //    the rows re-read from L1/L2
  // (threads t and t + 64 share token t's row, each half of its 16-byte pieces)
  {
    const float bt = sm.beta[t];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < dv / 16) {
        const int p = vp0 + i;
        float f[8];
        bf16x8(vpiece[i], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) *reinterpret_cast<float*>(sm.buf + sw_off(128, 8 * p + e, t)) = to_tf32(bt * f[e]);
      }
    }
  }
  to_async();
  mma_buf(64, at, kChunk, false);
  mma_wait();
  {
    const float sc = sm.beta[t] * sm.gam[t] * sm.rn[t];
    const int p0 = is_k ? 0 : DK / 16;
#pragma unroll 2
    for (int p = p0; p < p0 + DK / 16; ++p) {
      float f[8];
      bf16x8(valid_t ? __ldg(krow + p) : make_uint4(0, 0, 0, 0), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) *reinterpret_cast<float*>(sm.buf + sw_off(128, 8 * p + e, t)) = to_tf32(sc * f[e]);
    }
  }
  to_async();
  mma_buf(0, at, kChunk, false);
  mma_wait();
  // 6. W1^T rows into the buffer as the next A operand, W1 (token rows) out;
  //    then Oloc^T = W1^T Mq^T (TMEM 64..127)
  {
    const int r = tid;                  // TMEM lane = value row
    float* w1u = ws.w1 + u * kChunk * dv;
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      uint32_t r1[16];
      tmem_ld16(tmem + lane_base + 64 + q * 16, r1);
      tmem_ld_wait();
#pragma unroll
      for (int jj = 0; jj < 16; jj += 4) {
        const int j = q * 16 + jj;
        *reinterpret_cast<float4*>(sm.buf + sw_off(128, r, j)) =
            make_float4(to_tf32(__uint_as_float(r1[jj])), to_tf32(__uint_as_float(r1[jj + 1])),
                        to_tf32(__uint_as_float(r1[jj + 2])), to_tf32(__uint_as_float(r1[jj + 3])));
        if (r < dv) {
          // token rows: the warp's 32 value rows of one token are one 128-byte line
#pragma unroll
          for (int e = 0; e < 4; ++e) w1u[(j + e) * dv + r] = __uint_as_float(r1[jj + e]);
        }
      }
    }
  }
  to_async();
  mma_buf(64, mq, kChunk, false);
  mma_wait();
  // 7. Oloc (token rows) out; W2^T rows into the buffer and W2 into the bq
  //    image rows 0..63; then (Mq W2)^T = W2^T Mq^T (TMEM 0..63)
  {
    const int r = tid;
    float* olu = ws.ol + u * kChunk * dv;
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      uint32_t r1[16], r2[16];
      tmem_ld16(tmem + lane_base + 64 + q * 16, r1);
      tmem_ld16(tmem + lane_base + 0 + q * 16, r2);
      tmem_ld_wait();
      if (r < dv) {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) olu[(q * 16 + jj) * dv + r] = __uint_as_float(r1[jj]);
      }
#pragma unroll
      for (int jj = 0; jj < 16; jj += 4) {
        const int j = q * 16 + jj;
        float w2v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) w2v[e] = to_tf32(__uint_as_float(r2[jj + e]));
        *reinterpret_cast<float4*>(sm.buf + sw_off(128, r, j)) = make_float4(w2v[0], w2v[1], w2v[2], w2v[3]);
        if (r < DK) {
#pragma unroll
          for (int e = 0; e < 4; ++e) bq[sw_off(128, j + e, r) >> 2] = w2v[e];
        }
      }
    }
  }
  to_async();
  mma_buf(0, mq, kChunk, false);
  mma_wait();
  // 8. Qe = gamma q^ - Mq W2 into the bq image rows 64..127
  {
    const int r = tid;
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      uint32_t r1[16];
      tmem_ld16(tmem + lane_base + 0 + q * 16, r1);
      tmem_ld_wait();
      if (r < DK) {
        // all 16 loads before any store (one round trip)
        float gq[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) gq[jj] = __ldcg(bq + (sw_off(128, 64 + q * 16 + jj, r) >> 2));
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
          bq[sw_off(128, 64 + q * 16 + jj, r) >> 2] = to_tf32(gq[jj] - __uint_as_float(r1[jj]));
      }
    }
    if (tid == 0) ws.gc[u] = expf(GC);
  }
  fence_proxy_async_global();               // the bq and kd images are read by bulk copies
  tc_fence_before();
  gbar();
}

template <int DK>
__global__ void __launch_bounds__(kPrepThreads)
delta_prep_kernel(ScanArgs a, long long slots) {
  extern __shared__ uint8_t smem_raw[];
  PrepSmem<DK>& sm = *reinterpret_cast<PrepSmem<DK>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 1) { tmem_alloc(&sm.tmem_base, 128); tmem_relinquish(); }
  if (tid == 0) { mbar_init(&sm.bar, 1); fence_barrier_init(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  uint32_t phase = 0;
  bool ok = true;
  delta_prep_unit<DK>(a, slots, blockIdx.x, blockIdx.y, sm, tid, sm.tmem_base, phase, ok, 1);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(sm.tmem_base, 128);
}

// ---------------------------------------------------------------------------
// state carry
// ---------------------------------------------------------------------------
// The state is kept as S~ with S = Gamma S~ for a scalar Gamma carried from
// chunk to chunk, so that a chunk's decay gamma_C costs no pass over S:
//   U^T(MMA operand) = (W1^T - Gamma D1) / (gamma_C Gamma),  S~ += U^T Kd,
//   Gamma <- gamma_C Gamma,   O = Gamma D3 + Oloc.
// When gamma_C Gamma would drop below 2^-40 the chunk rescales S~ by it
// instead (after both products of the chunk have read S~) and Gamma restarts
// at 1.  Every role replays this recurrence on the same values, so all agree.
constexpr float kGammaFloor = 9.094947e-13f;   // 2^-40

__device__ __forceinline__ bool gamma_step(float gc, float& Gamma, float& inv) {
  const float p = gc * Gamma;
  if (p < kGammaFloor) {        // rescale S~ now: U^T unscaled, Gamma restarts
    inv = 1.f;
    Gamma = 1.f;
    return true;
  }
  inv = 1.f / p;
  Gamma = p;
  return false;
}

template <int DK>
struct ChainSmem {
  alignas(1024) uint8_t bq[2][128 * DK * 4];       // [W2; Qe] images
  alignas(1024) uint8_t kd[2][DK * kChunk * 4];    // Kd^T images
  alignas(16) uint16_t ostage[2][kChunk * 128];    // a chunk's bf16 outputs, [token][value row]
  uint64_t bq_full[2], kd_full[2], bq_empty[2], kd_empty[2], a1_done, a3_done[2], d_free[2], u_ready, init_ready, fin;
  uint64_t seen[8];                 // one-launch form: chunk c's unit seen complete by the copy issuer (slot c % 8)
  uint32_t tmem_base;
  int abort;
};

constexpr int kChainThreads2 = 320;   // warps 0-3 state, 4 copies, 5 MMA issue, 6-9 output

// The state carry of sequence b, value head h, by a whole CTA (warps 0..9;
// any further warps only take the CTA barriers).  With `fused` the per-chunk
// products are computed by other CTAs of the same launch, and every read of a
// unit waits for its flag.
template <int DK>
__device__ __forceinline__ void delta_chain_cta(const ScanArgs& a, long long slots, int b, int h, ChainSmem<DK>& sm,
                                                bool fused) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int dv = a.dv;
  const int t_seq0 = __ldg(a.cu_kept + b), t_seq1 = __ldg(a.cu_kept + b + 1);
  const int len = t_seq1 - t_seq0;
  if (len < 0 || t_seq0 < 0 || static_cast<long long>(t_seq1) > a.n_kept) {   // the same in every thread
    if (tid == 0) record_error(a.status, kStatusIndex);
    return;
  }
  const int nc = (len + kChunk - 1) / kChunk;
  const long long slot0 = t_seq0 / kChunk + b;
  const ChunkWs ws = chunk_ws(a.ws, slots, a.hv, DK, dv);
  const long long wd = a.watchdog;
  constexpr uint32_t kBqBytes = 128 * DK * 4, kKdBytes = DK * kChunk * 4;
  // chunk c's unit is complete.  The copy issuer polls the unit's flag (an
  // acquire at GPU scope) and then arrives on seen[c % 8]; the state and
  // output warps wait on that barrier (whole warps, the verdict the same in
  // every lane), which orders their loads of the unit after its stores
  // without a round trip to L2 on their path.  The issuer runs at most four
  // chunks ahead of the slowest of them (its copies of chunk c wait for the
  // output warps' release of chunk c - 4), so eight slots never alias.
  auto ready = [&](int c, bool warp_all) -> bool {
    if (!fused) return true;
    if (!warp_all) return flag_wait(ws.flag + (slot0 + c) * a.hv + h, wd, a.status);
    const bool r = mbar_wait(&sm.seen[c & 7], static_cast<uint32_t>(c >> 3) & 1u, wd, a.status, kStatusTimeout);
    return __all_sync(0xffffffffu, r);
  };

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.bq_full[s], 1);
      mbar_init(&sm.kd_full[s], 1);
      mbar_init(&sm.bq_empty[s], 1);
      mbar_init(&sm.kd_empty[s], 1);
      mbar_init(&sm.a3_done[s], 1);
      mbar_init(&sm.d_free[s], 4);
    }
    mbar_init(&sm.a1_done, 1);
    mbar_init(&sm.u_ready, 4);
    mbar_init(&sm.init_ready, 4);
    mbar_init(&sm.fin, 1);
    for (int s8 = 0; s8 < 8; ++s8) mbar_init(&sm.seen[s8], 1);
    sm.abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) { tmem_alloc(&sm.tmem_base, 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  // TMEM columns: S~ 0..127, D[0] 128..255, D[1] 256..383 (D1 the first 64
  // of each, D3 the second 64), U^T 384..447
  const uint32_t tS = tmem, tU = tmem + 384;
  auto tD = [&](int s) { return tmem + 128u + static_cast<uint32_t>(s) * 128u; };
  auto gc_of = [&](int c) { return __ldcg(ws.gc + (slot0 + c) * a.hv + h); };

  if (warp == 4) {
    // ---------------- operand copies ----------------
    // the [W2; Qe] image of a stage is free once the chunk's two first
    // products have read it, its Kd^T image once the state update has: each
    // is refilled as soon as it is free
    if (lane == 0) {
      int bq_issued = 0, kd_issued = 0;
      for (int c = 0; c < nc && !sm.abort; ++c) {
        const int s = c & 1;
        const long long u = (slot0 + c) * a.hv + h;
        if (!ready(c, false)) {
          sm.abort = 1;
          break;
        }
        if (fused) {
          fence_proxy_async_global();
          mbar_arrive(&sm.seen[c & 7]);
        }
        if (c >= 2 && !mbar_wait(&sm.bq_empty[s], ((c >> 1) - 1) & 1, wd, a.status, kStatusTimeout)) {
          sm.abort = 1;
          break;
        }
        mbar_arrive_expect_tx(&sm.bq_full[s], kBqBytes);
        bulk_copy_g2s(sm.bq[s], ws.bq + u * 128 * DK, kBqBytes, &sm.bq_full[s]);
        bq_issued = c + 1;
        if (c >= 2 && !mbar_wait(&sm.kd_empty[s], ((c >> 1) - 1) & 1, wd, a.status, kStatusTimeout)) {
          sm.abort = 1;
          break;
        }
        mbar_arrive_expect_tx(&sm.kd_full[s], kKdBytes);
        bulk_copy_g2s(sm.kd[s], ws.kd + u * DK * kChunk, kKdBytes, &sm.kd_full[s]);
        kd_issued = c + 1;
      }
      // every copy issued has landed before the CTA leaves (the earlier ones
      // were waited for by the MMA issuer before it freed their stages)
      for (int c2 = max(0, bq_issued - 2); c2 < bq_issued; ++c2)
        mbar_wait(&sm.bq_full[c2 & 1], (c2 >> 1) & 1, kDrainCycles, a.status, kStatusTimeout);
      for (int c2 = max(0, kd_issued - 2); c2 < kd_issued; ++c2)
        mbar_wait(&sm.kd_full[c2 & 1], (c2 >> 1) & 1, kDrainCycles, a.status, kStatusTimeout);
    }
  } else if (warp == 5) {
    // ---------------- MMA issue ----------------
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait_spin(bar, parity, wd, a.status, kStatusTimeout) && !sm.abort);
    };
    const uint32_t idesc_a = idesc_tf32_f32(128, 64);
    const uint32_t idesc_b = idesc_tf32_f32(128, DK);
    bool ok = nc > 0 && wait(&sm.init_ready, 0);
    bool any_mma = false;                    // an MMA was issued (then the final commit must cover it)
    for (int c = 0; ok && c < nc; ++c) {
      const int s = c & 1;
      if (!wait(&sm.bq_full[s], (c >> 1) & 1)) { ok = false; break; }
      if (c >= 2 && !wait(&sm.d_free[s], ((c >> 1) - 1) & 1)) { ok = false; break; }
      tc_fence_after();
      // D1 = S~ W2^T (the critical product), then D3 = S~ Qe^T (the output's)
      const uint64_t dw = smem_desc_sw128(smem_u32(sm.bq[s]), 16, 1024);
      const uint64_t dq = smem_desc_sw128(smem_u32(sm.bq[s]) + 64 * 128, 16, 1024);
      any_mma = true;
#pragma unroll
      for (int ks = 0; ks < DK / 8; ++ks)
        mma_tf32_ts_warp(tD(s), tS + ks * 8, dw + (sw_kstep(128, ks) >> 4), idesc_a, ks > 0 ? 1u : 0u);
      mma_commit_warp(&sm.a1_done);
#pragma unroll
      for (int ks = 0; ks < DK / 8; ++ks)
        mma_tf32_ts_warp(tD(s) + 64, tS + ks * 8, dq + (sw_kstep(128, ks) >> 4), idesc_a, ks > 0 ? 1u : 0u);
      mma_commit_warp(&sm.a3_done[s]);
      mma_commit_warp(&sm.bq_empty[s]);
      if (!wait(&sm.u_ready, c & 1)) { ok = false; break; }
      if (!wait(&sm.kd_full[s], (c >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      // S~ += U^T Kd
      const uint64_t dkd = smem_desc_sw128(smem_u32(sm.kd[s]), 16, 1024);
#pragma unroll
      for (int ks = 0; ks < kChunk / 8; ++ks)
        mma_tf32_ts_warp(tS, tU + ks * 8, dkd + (sw_kstep(DK, ks) >> 4), idesc_b, 1u);
      mma_commit_warp(&sm.kd_empty[s]);
    }
    if (!ok && nc > 0 && lane == 0) sm.abort = 1;
    if (any_mma || nc == 0) {
      // the final state (or, after an abort, the drain of the MMAs issued)
      mma_commit_warp(&sm.fin);
    } else if (lane == 0) {
      mbar_arrive(&sm.fin);
    }
  } else if (warp < 4) {
    // ---------------- state rows (warps 0..3) ----------------
    const int r = warp * 32 + lane;          // TMEM lane = value row
    const bool valid = r < dv;
    const uint32_t lb = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll
    for (int c0 = 0; c0 < DK; c0 += 32) {
      uint32_t v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0u;
      if (valid && a.initial_state) {
        const float* src = a.initial_state + ((static_cast<long long>(b) * a.hv + h) * dv + r) * DK + c0;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          const float4 f = __ldg(reinterpret_cast<const float4*>(src + j));
          v[j] = __float_as_uint(f.x); v[j + 1] = __float_as_uint(f.y);
          v[j + 2] = __float_as_uint(f.z); v[j + 3] = __float_as_uint(f.w);
        }
      }
      tmem_st32(tS + lb + c0, v);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.init_ready);
    // the W1^T row of the next chunk in registers; the one after it is
    // prefetched into L2, so that the register load hits L2
    float w[kChunk];
    auto w1_unit = [&](int c) { return ws.w1 + ((slot0 + c) * a.hv + h) * kChunk * dv; };
    auto fetch = [&](int c) {
      if (c >= nc || !valid) return;
      const float* src = w1_unit(c) + r;
#pragma unroll
      for (int j = 0; j < kChunk; ++j) w[j] = __ldcg(src + j * dv);
    };
    auto prefetch_l2 = [&](int c) {         // the unit's 64 x dv floats, two lines a thread
      if (c >= nc) return;
      const char* base = reinterpret_cast<const char*>(w1_unit(c));
      const int lines = kChunk * dv * 4 / 128;
      for (int l = warp * 32 + lane; l < lines; l += 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(base + l * 128));
    };
#pragma unroll
    for (int j = 0; j < kChunk; ++j) w[j] = 0.f;
    float Gamma = 1.f;
    bool ok = nc == 0 || ready(0, true);
    float gc_next = 1.f;
    if (ok && nc > 0) {
      fetch(0);
      gc_next = gc_of(0);
    }
    prefetch_l2(1);
    auto step = [&](int c) -> bool {
      const int s = c & 1;
      const float gc = gc_next;
      if (!mbar_wait(&sm.a1_done, c & 1, wd, a.status, kStatusTimeout) || sm.abort) return false;
      tc_fence_after();
      const float G0 = Gamma;
      float inv;
      const bool rescale = gamma_step(gc, Gamma, inv);
      // U^T = (W1^T - Gamma D1) / (gamma_C Gamma), into TMEM as the next A operand
      {
        // the four loads in flight together, one wait
        uint32_t d[4][16];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld16(tD(s) + lb + q * 16, d[q]);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            d[q][j] = __float_as_uint(to_tf32((w[q * 16 + j] - G0 * __uint_as_float(d[q][j])) * inv));
          tmem_st16(tU + lb + q * 16, d[q]);
        }
      }
      if (rescale) {
        // S~ <- gamma_C Gamma S~, once both products of the chunk have read it
        if (!mbar_wait(&sm.a3_done[s], (c >> 1) & 1, wd, a.status, kStatusTimeout)) return false;
        tc_fence_after();
        const float sc = gc * G0;
#pragma unroll
        for (int c0 = 0; c0 < DK; c0 += 16) {
          uint32_t sv[16];
          tmem_ld16(tS + lb + c0, sv);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) sv[j] = __float_as_uint(sc * __uint_as_float(sv[j]));
          tmem_st16(tS + lb + c0, sv);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.u_ready);
      if (c + 1 < nc) {                      // the registers take the next chunk's row
        if (!ready(c + 1, true)) return false;
        fetch(c + 1);
        gc_next = gc_of(c + 1);
      }
      prefetch_l2(c + 2);
      return true;
    };
    for (int c = 0; c < nc && ok; ++c) ok = step(c);
    if (!ok) sm.abort = 1;
    // the final state S = Gamma S~
    ok = mbar_wait(&sm.fin, 0, ok ? wd : kDrainCycles, a.status, kStatusTimeout) && ok;
    tc_fence_after();
    if (a.final_state) {
      float* dst = a.final_state + ((static_cast<long long>(b) * a.hv + h) * dv + (valid ? r : 0)) * DK;
#pragma unroll
      for (int c0 = 0; c0 < DK; c0 += 32) {
        uint32_t sv[32];
        tmem_ld32(tS + lb + c0, sv);
        tmem_ld_wait();
        if (valid && ok) {
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(dst + c0 + j) =
                make_float4(Gamma * __uint_as_float(sv[j]), Gamma * __uint_as_float(sv[j + 1]),
                            Gamma * __uint_as_float(sv[j + 2]), Gamma * __uint_as_float(sv[j + 3]));
        }
      }
    }
  } else if (warp < 10) {
    // ---------------- outputs (warps 6..9): O = Gamma D3 + Oloc ----------------
    const int q4 = warp & 3;                 // TMEM lane quadrant of this warp
    const int r = q4 * 32 + lane;
    const bool valid = r < dv;
    const uint32_t lb = static_cast<uint32_t>(q4 * 32) << 16;
    uint16_t* o = static_cast<uint16_t*>(a.o);
    float Gamma = 1.f;
    float ol[kChunk];
    auto ol_unit = [&](int c) { return ws.ol + ((slot0 + c) * a.hv + h) * kChunk * dv; };
    auto fetch = [&](int c) {
      if (c >= nc || !valid) return;
      const float* src = ol_unit(c) + r;
#pragma unroll
      for (int j = 0; j < kChunk; ++j) ol[j] = __ldcg(src + j * dv);
    };
#pragma unroll
    for (int j = 0; j < kChunk; ++j) ol[j] = 0.f;
    // every output warp takes the named barrier of every chunk, also after an
    // abort (work skipped, waits bounded), so that none waits on it forever
    bool dead = nc > 0 && !ready(0, true);
    if (dead) sm.abort = 1;
    float gc_next = 1.f;
    if (!dead && nc > 0) {
      fetch(0);
      gc_next = gc_of(0);
    }
    for (int c = 0; c < nc; ++c) {
      const int s = c & 1;
      const int n = min(kChunk, len - c * kChunk);
      uint16_t* stage = sm.ostage[c & 1];
      const float gc = gc_next;
      if (!dead) {
        if (!mbar_wait(&sm.a3_done[s], (c >> 1) & 1, wd, a.status, kStatusTimeout) || sm.abort) {
          sm.abort = 1;
          dead = true;
        } else {
          tc_fence_after();
          const float G0 = Gamma;
          float inv;
          gamma_step(gc, Gamma, inv);
          // D3 into registers, then D is released to the next-but-one
          // chunk's products before the stores
          uint32_t d3[kChunk];
          tmem_ld32(tD(s) + lb + 64, *reinterpret_cast<uint32_t(*)[32]>(&d3[0]));
          tmem_ld32(tD(s) + lb + 96, *reinterpret_cast<uint32_t(*)[32]>(&d3[32]));
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.d_free[s]);
          // the chunk's outputs through shared memory, so that they leave as
          // whole 16-byte pieces of token rows
          if (valid) {
#pragma unroll
            for (int j = 0; j < kChunk; ++j)
              stage[j * dv + r] =
                  static_cast<uint16_t>(pack_bf16x2(fmaf(G0, __uint_as_float(d3[j]), ol[j]), 0.f) & 0xFFFFu);
          }
        }
      }
      // the previous chunk's row copies have read their stage: after the
      // barrier every output thread may write the stage they read two chunks ago
      if (lane == 0) bulk_wait_read_0();
      fence_proxy_async_smem();
      asm volatile("bar.sync 2, 128;" ::: "memory");     // the four output warps
      if (!dead) {
        // the token rows leave by the bulk-copy engine, one copy per row, each
        // warp's lane 0 issuing every fourth row
        if (lane == 0) {
          for (int j = warp - 6; j < n; j += 4)
            bulk_copy_s2g(o + (static_cast<long long>(t_seq0 + c * kChunk + j) * a.hv + h) * dv, stage + j * dv,
                          static_cast<uint32_t>(dv) * 2u);
          bulk_commit_group();
        }
        if (c + 1 < nc) {
          if (ready(c + 1, true)) {
            fetch(c + 1);
            gc_next = gc_of(c + 1);
          } else {
            sm.abort = 1;
            dead = true;
          }
        }
        if (!dead && c + 2 < nc) {
          const char* base = reinterpret_cast<const char*>(ol_unit(c + 2));
          const int lines = kChunk * dv * 4 / 128;
          for (int l = (warp - 6) * 32 + lane; l < lines; l += 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(base + l * 128));
        }
      }
    }
    if (lane == 0) bulk_wait_0();          // the outputs are written before the CTA leaves
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

template <int DK>
__global__ void __launch_bounds__(kChainThreads2, 1)
delta_chain_kernel(ScanArgs a, long long slots) {
  extern __shared__ uint8_t smem_raw[];
  ChainSmem<DK>& sm = *reinterpret_cast<ChainSmem<DK>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  delta_chain_cta<DK>(a, slots, blockIdx.x, blockIdx.y, sm, false);
}

// ---------------------------------------------------------------------------
// both in one launch
// ---------------------------------------------------------------------------
constexpr int kFusedMaxBatch = 96;
constexpr long long kStaggerCycles = 235;   // per key dim: about a third of a unit's duration

// The chunks in the order (chunk index c within its sequence, then sequence
// b), the order in which the state carries of all sequences reach them.  Held
// by a whole warp (batch <= 96): lane keeps the start and the chunk count of
// sequences lane, lane + 32 and lane + 64.
struct ChunkOrder {
  int cu[3], nc[3];
  int max_nc;
  bool single;                              // one sequence: its chunks in order, no search
  __device__ __forceinline__ void init(const ScanArgs& a, int lane) {
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const int b = lane + 32 * i;
      cu[i] = 0;
      nc[i] = 0;
      if (b < a.batch) {
        cu[i] = __ldg(a.cu_kept + b);
        const int len = __ldg(a.cu_kept + b + 1) - cu[i];
        nc[i] = len > 0 ? (len + kChunk - 1) / kChunk : 0;
      }
    }
    max_nc = __reduce_max_sync(0xffffffffu, max(nc[0], max(nc[1], nc[2])));
    single = a.batch == 1;
    if (single) {                           // every lane holds sequence 0's start and count
      cu[0] = __shfl_sync(0xffffffffu, cu[0], 0);
      nc[0] = __shfl_sync(0xffffffffu, nc[0], 0);
    }
  }
  // the chunks ahead of chunk index c: the sum over b of min(nc_b, c)
  __device__ __forceinline__ long long ahead(int c) const {
    return static_cast<long long>(__reduce_add_sync(0xffffffffu, min(nc[0], c) + min(nc[1], c) + min(nc[2], c)));
  }
  // the slot of the q-th chunk, -1 past the last one
  __device__ __forceinline__ int slot(long long q) const {
    if (single) return q < nc[0] ? cu[0] / kChunk + static_cast<int>(q) : -1;
    if (q >= ahead(max_nc)) return -1;
    int lo = 0, hi = max_nc;                // ahead(lo) <= q < ahead(hi)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (ahead(mid) <= q) lo = mid; else hi = mid;
    }
    int j = static_cast<int>(q - ahead(lo));   // the j-th sequence with more than lo chunks
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      unsigned m = __ballot_sync(0xffffffffu, nc[i] > lo);
      const int cnt = __popc(m);
      if (j < cnt) {
        for (int t = 0; t < j; ++t) m &= m - 1;
        const int l = __ffs(m) - 1;
        const int b = 32 * i + l;
        return __shfl_sync(0xffffffffu, cu[i], l) / kChunk + b + lo;
      }
      j -= cnt;
    }
    return -1;
  }
};

// The state carry of a sequence walks its chunks one after another on one SM
// while the per-chunk products have no order among them, so one cooperative
// launch (every CTA resident, so that a CTA may wait for another) runs both
// side by side: CTAs 0 .. batch * hv - 1 carry the states, the others compute
// the units chunk index by chunk index (the order the chains consume them),
// three groups of four warps per CTA, each group with its own shared-memory
// share and 128 TMEM columns, and publish each finished unit by its flag.
// A group takes its next unit from a counter in the workspace (cleared with
// the flags), so that groups that started later take fewer units.
constexpr int kFusedThreads = 384;

template <int DK>
__global__ void __launch_bounds__(kFusedThreads, 1)
delta_fused_kernel(ScanArgs a, long long slots, int n_chain) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int cta = static_cast<int>(blockIdx.x);
  if (cta < n_chain) {
    delta_chain_cta<DK>(a, slots, cta / a.hv, cta % a.hv, *reinterpret_cast<ChainSmem<DK>*>(base), true);
    return;
  }
  PrepSmem<DK>* psm = reinterpret_cast<PrepSmem<DK>*>(base);
  const int tid = threadIdx.x, warp = tid >> 5, grp = warp >> 2, gtid = tid & 127;
  if (warp == 0) { tmem_alloc(&psm[0].tmem_base, 512); tmem_relinquish(); }
  if (gtid == 0) { mbar_init(&psm[grp].bar, 1); fence_barrier_init(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = psm[0].tmem_base + static_cast<uint32_t>(grp) * 128u;
  const ChunkWs ws = chunk_ws(a.ws, slots, a.hv, DK, a.dv);
  const long long units = slots * a.hv;
  uint32_t phase = 0;
  bool ok = true;
  ChunkOrder order;
  order.init(a, tid & 31);
  // the three groups of a CTA start a third of a unit apart, so that their
  // load, barrier and MMA phases interleave instead of coinciding
  if (grp > 0) {
    const long long t0 = clock64();
    while (clock64() - t0 < grp * kStaggerCycles * DK) __nanosleep(200);
  }
  // the unit counter, 8-byte aligned after the flags (the workspace base is
  // 256-byte aligned and every region before it a multiple of 256 bytes)
  unsigned long long* next = reinterpret_cast<unsigned long long*>(ws.flag + units);
  auto group_sync = [&]() { asm volatile("bar.sync %0, 128;" ::"r"(1 + 2 * grp) : "memory"); };
  if (gtid == 0) psm[grp].next_unit = static_cast<long long>(atomicAdd(next, 1ull));
  group_sync();
  long long k = psm[grp].next_unit;
  while (k < units) {
    const int x = order.slot(k / a.hv);                        // the same in every warp
    if (x < 0) break;                                          // and so are later k
    // a sequence outside the tokens (flagged by its state carry) can give a
    // slot past the workspace; no unit and no flag for it
    if (x < slots) {
      const int h = static_cast<int>(k % a.hv);
      delta_prep_unit<DK>(a, slots, x, h, psm[grp], gtid, tmem, phase, ok, 1 + 2 * grp);
      // the unit ends with a barrier of the group after every thread's stores
      if (gtid == 0) st_release_gpu(ws.flag + static_cast<long long>(x) * a.hv + h, 1);
    }
    // the next unit is taken only now, so that it goes to whichever group is
    // free first
    if (gtid == 0) psm[grp].next_unit = static_cast<long long>(atomicAdd(next, 1ull));
    group_sync();
    k = psm[grp].next_unit;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(psm[0].tmem_base, 512);
}

template <int DK>
static cudaError_t launch_chunked_dk(const ScanArgs& a, cudaStream_t st) {
  const long long slots = chunk_slots(a.n_kept, a.batch);
  const size_t prep_smem = sizeof(PrepSmem<DK>) + 1024;
  const size_t chain_smem = sizeof(ChainSmem<DK>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(delta_prep_kernel<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(prep_smem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(delta_chain_kernel<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(chain_smem));
  if (e != cudaSuccess) return e;
  const long long n_chain = static_cast<long long>(a.batch) * a.hv;
  const long long units = slots * a.hv;
  if (a.n_kept > 0 && n_chain <= a.num_sms / 2 && a.batch <= kFusedMaxBatch) {
    // one launch: a CTA per SM, the chains on the first, units on the rest
    const size_t fused_smem = std::max(sizeof(ChainSmem<DK>), 3 * sizeof(PrepSmem<DK>)) + 1024;
    e = cudaFuncSetAttribute(delta_fused_kernel<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(fused_smem));
    if (e != cudaSuccess) return e;
    const long long n_prep = std::min<long long>(a.num_sms - n_chain, (units + 2) / 3);
    // the flags and, after them, the unit counter
    e = cudaMemsetAsync(chunk_ws(a.ws, slots, a.hv, DK, a.dv).flag, 0, static_cast<size_t>(units + 2) * sizeof(int),
                        st);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(n_chain + n_prep));
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = fused_smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, delta_fused_kernel<DK>, a, slots, static_cast<int>(n_chain));
    // a device that cannot hold the grid at once (part of its SMs unavailable)
    // runs the same work as two launches below
    if (e != cudaErrorCooperativeLaunchTooLarge) return e;
    (void)cudaGetLastError();
  }
  if (a.n_kept > 0) {
    delta_prep_kernel<DK><<<dim3(static_cast<unsigned>(slots), static_cast<unsigned>(a.hv)), kPrepThreads, prep_smem,
                            st>>>(a, slots);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  delta_chain_kernel<DK><<<dim3(static_cast<unsigned>(a.batch), static_cast<unsigned>(a.hv)), kChainThreads2,
                           chain_smem, st>>>(a, slots);
  return cudaGetLastError();
}

cudaError_t launch_delta_scan_chunked(const ScanArgs& a, cudaStream_t st) {
  if (a.batch == 0 || a.hv == 0) return cudaSuccess;
  return a.dk == 128 ? launch_chunked_dk<128>(a, st) : launch_chunked_dk<64>(a, st);
}

}  // namespace tg
