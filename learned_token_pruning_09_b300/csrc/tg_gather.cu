// Gather of the kept rows (TokenGate's pruned forward: the layers above the
// gate run on the kept tokens only), staged through shared memory by the
// bulk-copy engine.  A CTA takes a contiguous range of kept slots; each of its
// threads owns one row-sized shared-memory slot and its mbarrier, and walks
// the range's rows t, t + slots, t + 2 slots, ...:
//   * checks the kept id (inside its sequence and inside x) and writes its
//     original position and score;
//   * bulk-copies the row from x into its slot (cp.async.bulk, completion
//     counted in bytes on the slot's barrier), and once it lands, bulk-copies
//     the slot out to x_kept.
// A warp issues 32 row copies with one instruction, so every row of a range
// that fits the slots is in flight at once, no register holds row data, and
// the copies read x once and write x_kept once.  Launched early behind the
// top-K (programmatic dependent launch), the kernel waits for the kept ids
// before reading anything.  The row copies need 16-byte aligned rows (d a
// multiple of 8, checked on the host).
#include "tg_common.cuh"

namespace tg {

constexpr int kGatherMaxSlots = 128;   // threads (one slot each) per CTA at most
constexpr int kGatherCtasPerSm = 2;    // leaves room beside a top-K CTA still running

__device__ __forceinline__ int find_seq(const int32_t* cu, int batch, long long i) {
  // largest b with cu[b] <= i  (cu ascending, cu[0] = 0)
  int lo = 0, hi = batch;   // answer in [0, batch)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<long long>(__ldg(cu + mid)) <= i) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst_smem)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, const void* src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               ::"l"(dst), "r"(smem_u32(src_smem)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Dynamic shared memory: one barrier per slot, then the slots (row_bytes each,
// 128-byte aligned).  blockDim.x >= slots; threads past the slots only idle.
__global__ void __launch_bounds__(kGatherMaxSlots)
gather_kernel(GatherArgs a, int slots, long long rows_per_cta, uint32_t slots_off) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int t = threadIdx.x;
  const bool copy_rows = a.x_kept != nullptr;
  const uint32_t row_bytes = copy_rows ? static_cast<uint32_t>(a.d) * 2 : 0u;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem_raw) + t;
  uint8_t* slot = smem_raw + slots_off + static_cast<size_t>(t) * row_bytes;
  if (copy_rows && t < slots) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  pdl_wait();     // launched early behind the top-K: its kept ids must be complete
  if (t >= slots) return;
  const long long i0 = static_cast<long long>(blockIdx.x) * rows_per_cta;
  const long long i1 = min(static_cast<long long>(a.n_kept), i0 + rows_per_cta);
  const long long n_total_kept = __ldg(a.cu_kept + a.batch);
  const uint8_t* x = static_cast<const uint8_t*>(a.x);
  uint8_t* y = static_cast<uint8_t*>(a.x_kept);
  uint32_t phase = 0;
  bool stored = false;   // a store from the slot may still be reading it
  for (long long i = i0 + t; i < i1; i += slots) {
    const long long r = __ldg(a.kept_idx + i);
    // x and s are read only for the outputs asked for (a call for positions
    // alone passes neither)
    const bool in_x = (!copy_rows && !a.s_kept) || (r >= 0 && r < a.n_rows);
    const bool copy = copy_rows && in_x;
    if (copy) {
      // the row's copy goes out first; the sequence bounds are checked while
      // it is in flight
      if (stored) bulk_wait_read_all();
      mbar_arrive_expect_tx(bar, row_bytes);
      bulk_load(slot, x + r * row_bytes, row_bytes, bar);
    }
    const int b = find_seq(a.cu_kept, a.batch, i);
    const int lo = __ldg(a.cu_seqlens + b);
    const int hi = __ldg(a.cu_seqlens + b + 1);
    const bool ok = in_x && i < n_total_kept && r >= lo && r < hi;
    if (!ok) record_error(a.status, kStatusIndex);
    if (ok && a.pos_kept) a.pos_kept[i] = static_cast<int32_t>(r - lo);
    if (ok && a.s_kept) a.s_kept[i] = __ldg(a.s + r);
    if (!copy) continue;
    if (!mbar_wait(bar, phase, a.watchdog, a.status, kStatusTimeout)) {
      // the copy is still waited for (bounded), so none is in flight when
      // the thread leaves; no further row is started
      mbar_wait(bar, phase, kDrainCycles, a.status, kStatusTimeout);
      break;
    }
    phase ^= 1u;
    if (ok) {
      bulk_store(y + i * static_cast<long long>(row_bytes), slot, row_bytes);
      bulk_commit();
      stored = true;
    }
  }
  if (stored) bulk_wait_all();   // x_kept is written before the thread leaves
}

cudaError_t launch_gather(const GatherArgs& a, cudaStream_t st) {
  if (a.n_kept == 0) return cudaSuccess;
  int dev = 0, max_optin = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e != cudaSuccess) return e;
  const size_t row_bytes = a.x_kept ? static_cast<size_t>(a.d) * 2 : 0;
  long long grid = min(static_cast<long long>(a.num_sms) * kGatherCtasPerSm, static_cast<long long>(a.n_kept));
  const long long rows_per_cta = (a.n_kept + grid - 1) / grid;
  grid = (a.n_kept + rows_per_cta - 1) / rows_per_cta;
  // slots: the range's rows, as many as fit kGatherCtasPerSm CTAs on an SM
  // (1 KB of each CTA's share is the system's)
  const size_t slots_off = kGatherMaxSlots * sizeof(uint64_t);
  const size_t budget = min(static_cast<size_t>(max_optin), static_cast<size_t>(per_sm) / kGatherCtasPerSm - 1024);
  long long slots = min(rows_per_cta, static_cast<long long>(kGatherMaxSlots));
  if (row_bytes) slots = min(slots, static_cast<long long>((budget - slots_off) / row_bytes));
  if (slots < 1) return cudaErrorInvalidConfiguration;
  const size_t smem = slots_off + static_cast<size_t>(slots) * row_bytes;
  e = cudaFuncSetAttribute(gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // programmatic dependent launch behind the previous kernel (the top-K)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>((slots + 31) / 32 * 32));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gather_kernel, a, static_cast<int>(slots), rows_per_cta,
                            static_cast<uint32_t>(slots_off));
}

}  // namespace tg
