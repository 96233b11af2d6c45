// C-ABI front end of libfa.so: argument checks, TMA tensor maps, kernel
// selection and launch, device status word. See include/fa.h for the contract.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "fa.h"
#include "fa_internal.h"
#include "sched_slots.h"

// Device status word (one per device that loads the library): kernels OR in
// fa::kDev* codes; fa_get_device_status() reads and clears it.
__device__ int g_fa_status;

// Tile-scheduler counters {next tile, CTAs done}, one pair per launch slot.
// A launch takes a free slot (fa::SlotTable: never used, or its last launch
// has finished, which an event recorded after that launch tells); its last
// CTA puts the pair back to zero. With kSchedSlots launches in flight on one
// device, the next one reuses the slot handed out longest ago and its stream
// waits for that slot's event first (SlotHold).
constexpr int kSchedSlots = 64;
__device__ unsigned int g_fa_sched[kSchedSlots][2];

namespace {

#ifdef FA_TEST_WITHHOLD_KV
// test build only (fa_test_set_withhold): the key block whose K tile the
// forward kernel's CTA 0 withholds, -1 for none
std::atomic<int> g_test_withhold{-1};
#endif

constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 256;   // key ranges of the split-KV forward, at most

struct DevInfo {
  bool ready = false;
  int sms = 0;
  int* status = nullptr;
  unsigned int* sched = nullptr;
  std::mutex slot_mu;                  // held from taking a slot to recording its event
  fa::SlotTable<kSchedSlots> slots;
  cudaEvent_t done_ev[kSchedSlots] = {};   // recorded on the stream after each slot's launch
};

std::mutex g_mu;
DevInfo g_dev[kMaxDevices];

int current_device(DevInfo** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FA_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_NO_DEVICE;
    }
    if (major != 10 || minor != 3) return FA_ERR_NO_DEVICE;  // kernels are built for sm_103a
    void* sym = nullptr;
    if (cudaGetSymbolAddress(&sym, g_fa_status) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_CUDA;
    }
    d.status = static_cast<int*>(sym);
    if (cudaGetSymbolAddress(&sym, g_fa_sched) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_CUDA;
    }
    d.sched = static_cast<unsigned int*>(sym);
    for (int i = 0; i < kSchedSlots; ++i) {
      if (cudaEventCreateWithFlags(&d.done_ev[i], cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        for (int j = 0; j < i; ++j) cudaEventDestroy(d.done_ev[j]);
        return FA_ERR_CUDA;
      }
    }
    d.sms = sms;
    d.ready = true;
  }
  *out = &d;
  return FA_OK;
}

// One persistent launch's hold on a scheduler slot, taken under the
// device's slot lock for the whole launch:
//   - a free slot is used as it is;
//   - when all kSchedSlots are held by launches in flight, the slot handed
//     out longest ago is reused and the stream first waits for its event
//     (cudaStreamWaitEvent: the GPU orders the two launches, the host does
//     not block);
//   - launched() records the slot's event after the launch went out.
// On a stream that is being captured into a graph no event is queried,
// waited for or recorded (a capture may not touch events from outside it,
// and the library does not see the graph's replays): the launch gets the
// next slot in turn, untracked, and replays must not overlap other launches
// of the library. sched() == nullptr: the stream wait could not be issued.
class SlotHold {
 public:
  SlotHold(DevInfo* dev, cudaStream_t stream) : dev_(dev), stream_(stream), lock_(dev->slot_mu) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
      cudaGetLastError();
      cs = cudaStreamCaptureStatusActive;
    }
    capturing_ = cs != cudaStreamCaptureStatusNone;
    if (capturing_) {
      slot_ = dev->slots.untracked();
      return;
    }
    slot_ = dev->slots.take(
        [dev](int i) {
          const cudaError_t q = cudaEventQuery(dev->done_ev[i]);
          if (q == cudaErrorNotReady) return false;
          if (q != cudaSuccess) cudaGetLastError();
          return true;
        },
        reused_);
    if (reused_ && cudaStreamWaitEvent(stream, dev->done_ev[slot_], 0) != cudaSuccess) {
      cudaGetLastError();
      slot_ = -1;   // still held by its previous launch
    }
  }
  unsigned int* sched() const { return slot_ < 0 ? nullptr : dev_->sched + 2 * slot_; }
  // the launch went out (ok) or failed
  void launched(bool ok) {
    if (slot_ < 0 || capturing_) return;
    if (!ok) {
      // a reused slot stays held by its previous launch, whose event stands
      if (!reused_) dev_->slots.release(slot_);
      return;
    }
    if (cudaEventRecord(dev_->done_ev[slot_], stream_) != cudaSuccess) cudaGetLastError();
  }

 private:
  DevInfo* dev_;
  cudaStream_t stream_;
  std::lock_guard<std::mutex> lock_;
  bool capturing_ = false;
  bool reused_ = false;
  int slot_ = -1;
};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// 2-D map over a [rows, cols] row-major matrix, boxes of box_rows x box_cols,
// 128-byte swizzle (the layout the tcgen05 descriptors expect), zero fill
// outside the matrix.
int make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, uint64_t cols,
             uint64_t rows, uint32_t box_cols, uint32_t box_rows,
             CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (!fn) return FA_ERR_CUDA;
  cuuint64_t dims[2] = {cols, rows < 1 ? 1 : rows};
  cuuint64_t strides[1] = {cols * (uint64_t)elem_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Heads per tile group (fa::tile_order). Causal problems: as many heads as
// keep the streamed side of the group (two tensors of stream_rows x D
// elements per head) within about 32 MB of L2, 1 to 16; otherwise 1 (every
// tile of a head costs the same, head by head keeps the L2 footprint least).
int head_group(bool causal, int64_t BH, int64_t stream_rows, int D, int elem_bytes) {
  if (!causal) return 1;
  const int64_t per_head = std::max<int64_t>(stream_rows * D * elem_bytes * 2, 1);
  const int64_t fit = ((int64_t)32 << 20) / per_head;
  return (int)std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(BH, 16), fit));
}

}  // namespace

extern "C" {

#ifdef FA_TEST_WITHHOLD_KV
// test build only: later 16-bit forward launches withhold the K tile of key
// block kb in CTA 0's first work tile (kb < 0: none). Not in fa.h and not in
// the release library.
void fa_test_set_withhold(int kb) { g_test_withhold.store(kb); }
#endif

int fa_version(void) { return (1 << 16) | 4; }

const char* fa_strerror(int s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case FA_ERR_CUDA: return "CUDA call failed";
    case FA_ERR_DEVICE_TIMEOUT: return "device wait timed out; outputs incomplete";
    case FA_ERR_DEVICE_SEQLENS: return "cu_seqlens entry out of bounds; sequence skipped";
    case FA_ERR_NO_DEVICE: return "no sm_103 device is current";
    case FA_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the built-in 64 MiB array holds";
    case FA_ERR_BUSY: return "no scheduler slot could be given to the launch (the stream could not wait for one)";
    default: return "unknown status";
  }
}

}  // extern "C"

namespace {

// Argument checks and launch description shared by the 16-bit entry points
// (everything but the split-KV fields). Returns FA_OK, or the status to
// report; `nothing` is set when the problem is empty.
int setup_fwd16(fa::FwdLaunch& L, DevInfo** devp, bool* nothing, const void* q, const void* k,
                const void* v, void* o, float* lse, int B, int H, int Sq, int Sk, int D, float scale,
                int causal, const int* cu_seqlens_q, const int* cu_seqlens_k, int total_q, int total_k,
                int dtype, void* stream) {
  *nothing = false;
  // ---- host-side argument checks (no device access)
  if (dtype == FA_FP8_E4M3) return FA_ERR_UNSUPPORTED;
  if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
  if (B < 0 || H <= 0 || Sq < 0 || Sk < 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.f) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  const bool varlen = cu_seqlens_q != nullptr || cu_seqlens_k != nullptr;
  if (varlen && (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr)) return FA_ERR_INVALID_ARG;
  if (varlen && (total_q < 0 || total_k < 0)) return FA_ERR_INVALID_ARG;
  const int64_t Tq = varlen ? total_q : (int64_t)B * Sq;
  const int64_t Tk = varlen ? total_k : (int64_t)B * Sk;
  if (Tq > INT32_MAX || Tk > INT32_MAX) return FA_ERR_INVALID_ARG;
  if ((int64_t)H * D * 2 > (int64_t)1 << 38) return FA_ERR_INVALID_ARG;
  if (B == 0 || Tq == 0 || Sq == 0) {  // nothing to compute
    *nothing = true;
    return FA_OK;
  }
  // no keys at all: every row sees none, and the kernel's empty work tiles
  // write O = 0 and LSE = -inf; K and V are never read, so (possibly null,
  // as empty tensors are) their maps may point at O
  if (Tk == 0) k = v = o;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FA_ERR_ALIGNMENT;
  const int rows = fa::cta_rows16(D, Sq);
  const int64_t n_qblk = ((int64_t)Sq + rows - 1) / rows;
  const int64_t ntiles = (int64_t)B * H * n_qblk;
  if (ntiles > INT32_MAX || (int64_t)B * H * Sq > ((int64_t)1 << 40)) return FA_ERR_INVALID_ARG;

  // ---- device
  DevInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st != FA_OK) return st;
  *devp = dev;

  std::memset(&L, 0, sizeof(L));
  const CUtensorMapDataType dt = dtype == FA_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t cols = (uint64_t)H * D;
  if ((st = make_map(&L.tq, q, dt, 2, cols, (uint64_t)Tq, 64, 128)) != FA_OK) return st;
  if ((st = make_map(&L.tk, k, dt, 2, cols, (uint64_t)Tk, 64, 128)) != FA_OK) return st;
  if ((st = make_map(&L.tv, v, dt, 2, cols, (uint64_t)Tk, 64, 128)) != FA_OK) return st;
  if ((st = make_map(&L.to, o, dt, 2, cols, (uint64_t)Tq, 64, 128)) != FA_OK) return st;
  L.p.o = o;
  L.p.lse = lse;
  L.p.cu_q = cu_seqlens_q;
  L.p.cu_k = cu_seqlens_k;
  L.p.B = B;
  L.p.H = H;
  L.p.Sq = Sq;
  L.p.Sk = Sk;
  L.p.total_q = (int)Tq;
  L.p.total_k = (int)Tk;
  L.p.n_qblk = (int)n_qblk;
  L.p.ntiles = (int)ntiles;
  L.p.c = (float)((double)scale * 1.4426950408889634);
  L.p.status = dev->status;
  L.p.n_split = 1;
  L.p.split_blocks = 1 << 30;
#ifdef FA_TEST_WITHHOLD_KV
  L.p.test_withhold_kb = g_test_withhold.load();
#endif
  L.D = D;
  L.kind = dtype == FA_FP16 ? fa::kF16 : fa::kBF16;
  L.causal = causal != 0;
  L.one_tile = D <= 128 && rows == 128;
  L.num_sms = dev->sms;
  L.stream = static_cast<cudaStream_t>(stream);
  return FA_OK;
}

int launch16(fa::FwdLaunch& L, DevInfo* dev) {
  SlotHold hold(dev, L.stream);
  if ((L.p.sched = hold.sched()) == nullptr) return FA_ERR_BUSY;
  L.p.head_group = head_group(L.causal, (int64_t)L.p.B * L.p.H, L.p.Sk, L.D, 2);
  cudaError_t e;
  switch (L.D) {
    case 64: e = L.one_tile ? fa::launch_fwd_d64_q1(L) : fa::launch_fwd_d64(L); break;
    case 128: e = L.one_tile ? fa::launch_fwd_d128_q1(L) : fa::launch_fwd_d128(L); break;
    default: e = fa::launch_fwd_d256(L); break;
  }
  hold.launched(e == cudaSuccess);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

// Key ranges of the split-KV forward. `requested` > 0 asks for that many;
// `requested` <= 0 picks the count with the least estimated time, in units of
// one SM's time for one 128-key block: whole waves of work tiles over the SMs
// times (the blocks of one tile + about four blocks of per-tile overhead: Q
// load, pipeline fill, output write; two more when the tile writes an fp32
// partial O), plus, with more than one range, the merge, which moves every
// range's partial O twice (written, then read) at about 12 MB of HBM traffic
// per block time. Fewer ranges on ties. Work tiles come in whole waves, so 9
// ranges of 57 blocks in one wave beat 10 ranges in two; a prefill whose
// tiles already fill the SMs keeps one range, since the partials and their
// merge cost more than the last wave's idle SMs.
// Returns the ranges actually used (every range non-empty) and their length
// in 128-key blocks.
void resolve_splits(int B, int H, int Sq, int Sk, int D, int requested, int sms, int* n_split,
                    int* split_blocks) {
  const int64_t nblocks = ((int64_t)Sk + 127) / 128;
  const int rows = fa::cta_rows16(D, Sq);
  const int64_t tiles = (int64_t)B * H * (((int64_t)Sq + rows - 1) / rows);
  int64_t n = requested;
  if (n <= 0) {
    n = 1;
    if (tiles > 0 && sms > 0) {
      const int64_t kOverhead = 4, kPartialOverhead = 2;
      const int64_t kMergeBytesPerBlock = (int64_t)12 << 20;
      const int64_t partial_bytes = (int64_t)B * H * Sq * D * (int64_t)sizeof(float);   // one range's O
      int64_t best = -1;
      const int64_t top = nblocks < kMaxSplits ? nblocks : kMaxSplits;
      for (int64_t c = 1; c <= top; ++c) {
        const int64_t per = (nblocks + c - 1) / c;
        const int64_t used = (nblocks + per - 1) / per;   // non-empty ranges
        if (used != c) continue;
        const int64_t waves = (tiles * c + sms - 1) / sms;
        int64_t cost = waves * (per + kOverhead + (c > 1 ? kPartialOverhead : 0));
        if (c > 1) cost += (2 * c * partial_bytes + kMergeBytesPerBlock - 1) / kMergeBytesPerBlock;
        if (best < 0 || cost < best) {
          best = cost;
          n = c;
        }
      }
    }
  }
  if (n > kMaxSplits) n = kMaxSplits;
  if (n > nblocks) n = nblocks;
  if (n < 1) n = 1;
  const int64_t per = (nblocks + n - 1) / n;
  *split_blocks = (int)(per < 1 ? 1 : per);
  *n_split = (int)(per < 1 ? 1 : (nblocks + per - 1) / per);
}

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace of the split-KV forward: partial O (fp32) then partial LSE.
size_t splitkv_bytes(int B, int H, int Sq, int D, int n_split) {
  return round256((size_t)n_split * B * Sq * H * D * sizeof(float)) + (size_t)n_split * B * H * Sq * sizeof(float);
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Sq,
           int Sk, int D, float scale, int causal, const int* cu_seqlens_q, const int* cu_seqlens_k,
           int total_q, int total_k, int dtype, void* stream) {
  fa::FwdLaunch L;
  DevInfo* dev = nullptr;
  bool nothing = false;
  int st = setup_fwd16(L, &dev, &nothing, q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, cu_seqlens_q,
                       cu_seqlens_k, total_q, total_k, dtype, stream);
  if (st != FA_OK || nothing) return st;
  return launch16(L, dev);
}

size_t fa_fwd_splitkv_workspace_size(int B, int H, int Sq, int Sk, int D, int num_splits) {
  if (B <= 0 || H <= 0 || Sq <= 0 || Sk < 0 || (D != 64 && D != 128 && D != 256)) return 0;
  int sms = 0;
  if (num_splits <= 0) {
    DevInfo* dev = nullptr;
    if (current_device(&dev) != FA_OK) return 0;
    sms = dev->sms;
  }
  int n = 1, per = 1;
  resolve_splits(B, H, Sq, Sk, D, num_splits, sms, &n, &per);
  return splitkv_bytes(B, H, Sq, D, n);
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Sq,
                   int Sk, int D, float scale, int causal, int num_splits, void* workspace,
                   size_t workspace_bytes, int dtype, void* stream) {
  fa::FwdLaunch L;
  DevInfo* dev = nullptr;
  bool nothing = false;
  int st = setup_fwd16(L, &dev, &nothing, q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, nullptr, nullptr,
                       0, 0, dtype, stream);
  if (st != FA_OK || nothing) return st;
  int n = 1, per = 1;
  resolve_splits(B, H, Sq, Sk, D, num_splits, dev->sms, &n, &per);
  const size_t need = splitkv_bytes(B, H, Sq, D, n);
  if (workspace == nullptr || workspace_bytes < need) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_ALIGNMENT;
  const int64_t ntiles = (int64_t)L.p.ntiles * n;
  if (ntiles > INT32_MAX) return FA_ERR_INVALID_ARG;
  L.p.ntiles = (int)ntiles;
  L.p.n_split = n;
  L.p.split_blocks = per;
  L.p.o_part = static_cast<float*>(workspace);
  L.p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                          round256((size_t)n * B * Sq * H * D * sizeof(float)));
  if ((st = launch16(L, dev)) != FA_OK) return st;
  cudaError_t e = fa::launch_splitkv_merge(L.p.o_part, L.p.lse_part, o, lse, n, B, H, Sq, D,
                                           dtype == FA_FP16, dev->sms, L.stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

int fa_fwd_paged(const void* q, const void* k_cache, const void* v_cache, const int* block_table,
                 const int* seqlens_k, void* o, float* lse, int B, int H, int Sq, int D, int num_pages,
                 int page_size, int max_pages, float scale, int causal, const int* cu_seqlens_q, int total_q,
                 int num_splits, void* workspace, size_t workspace_bytes, int dtype, void* stream) {
  // ---- host-side checks of the paging arguments (the rest: setup_fwd16)
  if (num_pages <= 0 || max_pages <= 0 || B < 0) return FA_ERR_INVALID_ARG;
  if (!(page_size == 16 || page_size == 32 || page_size == 64 || (page_size > 0 && page_size % 128 == 0)))
    return FA_ERR_INVALID_ARG;
  if ((int64_t)num_pages * page_size + 128 > INT32_MAX) return FA_ERR_INVALID_ARG;
  if ((int64_t)max_pages * page_size > INT32_MAX) return FA_ERR_INVALID_ARG;
  if ((int64_t)B * max_pages > INT32_MAX) return FA_ERR_INVALID_ARG;
  const int Sk = max_pages * page_size;   // the most keys a sequence can have
  if (B > 0 && (!block_table || !seqlens_k)) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(block_table) & 3u || reinterpret_cast<uintptr_t>(seqlens_k) & 3u)
    return FA_ERR_ALIGNMENT;
  // packed queries: one launch (the key-range merge assumes fixed lengths)
  const bool varlen_q = cu_seqlens_q != nullptr;
  if (varlen_q && num_splits != 1) return FA_ERR_UNSUPPORTED;
  if (varlen_q && total_q < 0) return FA_ERR_INVALID_ARG;
  fa::FwdLaunch L;
  DevInfo* dev = nullptr;
  bool nothing = false;
  // the contiguous setup (queries fixed-length or packed; the packed form
  // passes cu_seqlens_q for both sides, since the key side's offsets are
  // unused here); the K/V maps are replaced below by maps over the caches
  int st = setup_fwd16(L, &dev, &nothing, q, k_cache, v_cache, o, lse, B, H, Sq, 0, D, scale, causal,
                       cu_seqlens_q, cu_seqlens_q, varlen_q ? total_q : 0, 0, dtype, stream);
  if (st != FA_OK || nothing) return st;
  L.p.cu_k = nullptr;
  const CUtensorMapDataType dt = dtype == FA_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t cols = (uint64_t)H * D, rows = (uint64_t)num_pages * page_size;
  const uint32_t box_rows = page_size < 128 ? (uint32_t)page_size : 128u;
  if ((st = make_map(&L.tk, k_cache, dt, 2, cols, rows, 64, box_rows)) != FA_OK) return st;
  if ((st = make_map(&L.tv, v_cache, dt, 2, cols, rows, 64, box_rows)) != FA_OK) return st;
  L.p.Sk = Sk;
  L.p.total_k = (int)rows;
  L.p.block_table = block_table;
  L.p.seqlens_k = seqlens_k;
  L.p.max_pages = max_pages;
  L.p.page_size = page_size;
  L.p.num_pages = num_pages;
  L.p.page_rows = (int)box_rows;
  L.p.page_shift = (page_size & (page_size - 1)) == 0 ? __builtin_ctz((unsigned)page_size) : -1;
  L.p.n_kblk_tag = Sk / 128 + 2;
  if ((int64_t)B * L.p.n_kblk_tag > INT32_MAX) return FA_ERR_INVALID_ARG;
  int n = 1, per = 1;
  resolve_splits(B, H, Sq, Sk, D, num_splits, dev->sms, &n, &per);
  if (num_splits == 1) n = 1;
  if (n == 1) {
    L.p.split_blocks = 1 << 30;
    return launch16(L, dev);
  }
  const size_t need = splitkv_bytes(B, H, Sq, D, n);
  if (workspace == nullptr || workspace_bytes < need) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_ALIGNMENT;
  const int64_t ntiles = (int64_t)L.p.ntiles * n;
  if (ntiles > INT32_MAX) return FA_ERR_INVALID_ARG;
  L.p.ntiles = (int)ntiles;
  L.p.n_split = n;
  L.p.split_blocks = per;
  L.p.o_part = static_cast<float*>(workspace);
  L.p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                          round256((size_t)n * B * Sq * H * D * sizeof(float)));
  if ((st = launch16(L, dev)) != FA_OK) return st;
  cudaError_t e = fa::launch_splitkv_merge(L.p.o_part, L.p.lse_part, o, lse, n, B, H, Sq, D,
                                           dtype == FA_FP16, dev->sms, L.stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // extern "C"

namespace {

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// FP8 preparation, fixed length (cu_* == nullptr; Sq, Sk per sequence) or
// varlen (cu_seqlens_*, cu_blocks_*, totals; Sq, Sk = max lengths).
int prep_impl(const void* q, const void* k, const void* v, int in_dtype, void* q8, void* k8, void* v8,
              float* q_scale, float* k_scale, float* v_scale, const signed char* sigma, int B, int H, int Sq, int Sk,
              int D, const int* cu_q, const int* cu_k, const int* cbq, const int* cbk, int total_q, int total_k,
              void* stream) {
  if (in_dtype != FA_FP16 && in_dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if (D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
  if (B < 0 || H <= 0 || Sq < 0 || Sk < 0 || total_q < 0 || total_k < 0) return FA_ERR_INVALID_ARG;
  const bool varlen = cu_q != nullptr || cu_k != nullptr;
  if (!varlen && ((int64_t)B * Sq > INT32_MAX || (int64_t)B * Sk > INT32_MAX)) return FA_ERR_INVALID_ARG;
  if (B == 0 || (Sq == 0 && Sk == 0)) return FA_OK;
  const bool has_q = Sq > 0, has_kv = Sk > 0;
  if ((has_q && (!q || !q8 || !q_scale)) || (has_kv && (!k || !v || !k8 || !v8 || !k_scale || !v_scale)))
    return FA_ERR_INVALID_ARG;
  if (varlen && ((has_q && (!cu_q || !cbq)) || (has_kv && (!cu_k || !cbk)))) return FA_ERR_INVALID_ARG;
  for (const void* p : {q, k, v, (const void*)q8, (const void*)k8, (const void*)v8})
    if (p && !aligned16(p)) return FA_ERR_ALIGNMENT;
  for (const void* p : {(const void*)q_scale, (const void*)k_scale, (const void*)v_scale})
    if (p && !aligned4(p)) return FA_ERR_ALIGNMENT;
  DevInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st != FA_OK) return st;
  fa::PrepParams t[3] = {};
  int n = 0;
  auto add = [&](const void* x, void* x8, float* sc, const signed char* sg, int S, const int* cu, const int* cb,
                 int total) {
    fa::PrepParams& P = t[n++];
    P.x = x;
    P.x8 = static_cast<uint8_t*>(x8);
    P.scale = sc;
    P.sigma = reinterpret_cast<const int8_t*>(sg);
    P.B = B;
    P.H = H;
    P.S = S;
    P.nblk = (S + 127) / 128;
    P.bf16 = in_dtype == FA_BF16;
    P.cu_seqlens = cu;
    P.cu_blocks = cb;
    P.total = total;
    P.status = dev->status;
  };
  if (has_q) add(q, q8, q_scale, sigma, Sq, cu_q, cbq, total_q);
  if (has_kv) {
    add(k, k8, k_scale, sigma, Sk, cu_k, cbk, total_k);
    add(v, v8, v_scale, nullptr, Sk, cu_k, cbk, total_k);
  }
  // one [rows, H * D] map per tensor: the input in 64-element boxes with the
  // 128-byte swizzle (a thread reads its row across the banks), the e4m3
  // output in boxes of min(D, 128) bytes x 128 rows (64- or 128-byte swizzle)
  CUtensorMap in_maps[3], out_maps[3];
  const CUtensorMapDataType dt = in_dtype == FA_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  for (int i = 0; i < n; ++i) {
    const uint64_t rows = t[i].cu_seqlens != nullptr ? (uint64_t)t[i].total : (uint64_t)t[i].B * t[i].S;
    const uint64_t cols = (uint64_t)H * D;
    if ((st = make_map(&in_maps[i], t[i].x, dt, 2, cols, rows, 64, 128)) != FA_OK) return st;
    if ((st = make_map(&out_maps[i], t[i].x8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, cols, rows, D == 64 ? 64u : 128u,
                       128, D == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B)) != FA_OK)
      return st;
  }
  cudaError_t e = fa::launch_fp8_prep(t, in_maps, out_maps, n, D, dev->sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

int fwd_fp8_impl(const void* q8, const void* k8, const void* v8, const float* q_scale, const float* k_scale,
                 const float* v_scale, void* o, float* lse, int B, int H, int Sq, int Sk, int D, float scale,
                 int causal, const int* cu_q, const int* cu_k, const int* cbq, const int* cbk, int total_q,
                 int total_k, void* stream) {
  if (D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
  if (B < 0 || H <= 0 || Sq < 0 || Sk < 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.f) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  const bool varlen = cu_q != nullptr || cu_k != nullptr;
  if (varlen && (!cu_q || !cu_k || !cbq || !cbk || total_q < 0 || total_k < 0)) return FA_ERR_INVALID_ARG;
  const int64_t Tq = varlen ? total_q : (int64_t)B * Sq, Tk = varlen ? total_k : (int64_t)B * Sk;
  if (Tq > INT32_MAX || Tk > INT32_MAX) return FA_ERR_INVALID_ARG;
  if (B == 0 || Sq == 0 || Tq == 0) return FA_OK;
  // no keys at all: the empty work tiles write O = 0 and LSE = -inf and read
  // neither K, V nor their scales, so (possibly null) K and V may point at O
  if (Tk == 0) k8 = v8 = o;
  if (!q8 || !k8 || !v8 || !o || !lse || !q_scale || (Tk > 0 && (!k_scale || !v_scale)))
    return FA_ERR_INVALID_ARG;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8) || !aligned16(o) || !aligned4(lse) ||
      !aligned4(q_scale) || !aligned4(k_scale) || !aligned4(v_scale))
    return FA_ERR_ALIGNMENT;
  const int rows = fa::cta_rows(D);
  const int64_t n_qblk = ((int64_t)Sq + rows - 1) / rows;
  const int64_t ntiles = (int64_t)B * H * n_qblk;
  if (ntiles > INT32_MAX || (int64_t)B * H * Sq > ((int64_t)1 << 40)) return FA_ERR_INVALID_ARG;
  DevInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st != FA_OK) return st;

  fa::FwdLaunch L;
  std::memset(&L, 0, sizeof(L));
  const uint64_t cols = (uint64_t)H * D;
  const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  // boxes of 128 rows x 128 bytes (128-byte swizzle), or of one whole
  // 64-byte row (64-byte swizzle) at D = 64
  const uint32_t box = D == 64 ? 64u : 128u;
  const CUtensorMapSwizzle sw = D == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  if ((st = make_map(&L.tq, q8, dt, 1, cols, (uint64_t)Tq, box, 128, sw)) != FA_OK) return st;
  if ((st = make_map(&L.tk, k8, dt, 1, cols, (uint64_t)Tk, box, 128, sw)) != FA_OK) return st;
  if ((st = make_map(&L.tv, v8, dt, 1, cols, (uint64_t)Tk, box, 128, sw)) != FA_OK) return st;
  if ((st = make_map(&L.to, o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cols, (uint64_t)Tq, 64, 128)) != FA_OK)
    return st;
  L.p.o = o;
  L.p.lse = lse;
  L.p.cu_q = cu_q;
  L.p.cu_k = cu_k;
  L.p.cu_blocks_q = cbq;
  L.p.cu_blocks_k = cbk;
  L.p.B = B;
  L.p.H = H;
  L.p.Sq = Sq;
  L.p.Sk = Sk;
  L.p.total_q = (int)Tq;
  L.p.total_k = (int)Tk;
  L.p.n_qblk = (int)n_qblk;
  L.p.ntiles = (int)ntiles;
  L.p.c = (float)((double)scale * 1.4426950408889634);
  L.p.status = dev->status;
  L.p.n_split = 1;
  L.p.split_blocks = 1 << 30;
  L.p.q_scale = q_scale;
  L.p.k_scale = k_scale;
  L.p.v_scale = v_scale;
  L.p.nblk_q = (Sq + 127) / 128;
  L.p.nblk_k = (Sk + 127) / 128;
#ifdef FA_TEST_WITHHOLD_KV
  L.p.test_withhold_kb = -1;
#endif
  L.D = D;
  L.kind = fa::kE4M3;
  L.causal = causal != 0;
  L.p.head_group = head_group(L.causal, (int64_t)B * H, Sk, D, 1);
  L.num_sms = dev->sms;
  L.stream = static_cast<cudaStream_t>(stream);
  SlotHold hold(dev, L.stream);
  if ((L.p.sched = hold.sched()) == nullptr) return FA_ERR_BUSY;
  cudaError_t e = D == 64    ? fa::launch_fwd_fp8_d64(L)
                  : D == 128 ? fa::launch_fwd_fp8_d128(L)
                             : fa::launch_fwd_fp8_d256(L);
  hold.launched(e == cudaSuccess);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // namespace

extern "C" {

int fa_fp8_prep(const void* q, const void* k, const void* v, int in_dtype, void* q8, void* k8, void* v8,
                float* q_scale, float* k_scale, float* v_scale, const signed char* sigma, int B, int H,
                int Sq, int Sk, int D, void* stream) {
  return prep_impl(q, k, v, in_dtype, q8, k8, v8, q_scale, k_scale, v_scale, sigma, B, H, Sq, Sk, D, nullptr,
                   nullptr, nullptr, nullptr, 0, 0, stream);
}

int fa_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* q_scale, const float* k_scale,
               const float* v_scale, void* o, float* lse, int B, int H, int Sq, int Sk, int D, float scale,
               int causal, void* stream) {
  return fwd_fp8_impl(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, B, H, Sq, Sk, D, scale, causal, nullptr,
                      nullptr, nullptr, nullptr, 0, 0, stream);
}

int fa_varlen_blocks(const int* cu_seqlens, int B, int* cu_blocks, void* stream) {
  if (B < 0 || (B > 0 && (!cu_seqlens || !cu_blocks))) return FA_ERR_INVALID_ARG;
  DevInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st != FA_OK) return st;
  if (fa::launch_varlen_blocks(cu_seqlens, B, cu_blocks, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

int fa_fp8_prep_varlen(const void* q, const void* k, const void* v, int in_dtype, void* q8, void* k8, void* v8,
                       float* q_scale, float* k_scale, float* v_scale, const signed char* sigma, int B, int H,
                       const int* cu_seqlens_q, const int* cu_seqlens_k, const int* cu_blocks_q,
                       const int* cu_blocks_k, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                       int D, void* stream) {
  if ((max_seqlen_q > 0 && !cu_seqlens_q) || (max_seqlen_k > 0 && !cu_seqlens_k)) return FA_ERR_INVALID_ARG;
  return prep_impl(q, k, v, in_dtype, q8, k8, v8, q_scale, k_scale, v_scale, sigma, B, H, max_seqlen_q,
                   max_seqlen_k, D, cu_seqlens_q, cu_seqlens_k, cu_blocks_q, cu_blocks_k, total_q, total_k, stream);
}

int fa_fwd_fp8_varlen(const void* q8, const void* k8, const void* v8, const float* q_scale, const float* k_scale,
                      const float* v_scale, void* o, float* lse, int B, int H, const int* cu_seqlens_q,
                      const int* cu_seqlens_k, const int* cu_blocks_q, const int* cu_blocks_k, int total_q,
                      int total_k, int max_seqlen_q, int max_seqlen_k, int D, float scale, int causal,
                      void* stream) {
  if (!cu_seqlens_q || !cu_seqlens_k || !cu_blocks_q || !cu_blocks_k) return FA_ERR_INVALID_ARG;
  return fwd_fp8_impl(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, B, H, max_seqlen_q, max_seqlen_k, D, scale,
                      causal, cu_seqlens_q, cu_seqlens_k, cu_blocks_q, cu_blocks_k, total_q, total_k, stream);
}

size_t fa_bwd_workspace_size(int H, int total_q) {
  if (H <= 0 || total_q <= 0) return 0;
  return round256((size_t)2 * (size_t)H * (size_t)total_q * sizeof(float));
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
           void* dq, void* dk, void* dv, int B, int H, int Sq, int Sk, int D, float scale, int causal,
           const int* cu_seqlens_q, const int* cu_seqlens_k, int total_q, int total_k, void* workspace,
           size_t workspace_bytes, int dtype, void* stream) {
  // ---- host-side argument checks (no device access)
  if (dtype == FA_FP8_E4M3) return FA_ERR_UNSUPPORTED;
  if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
  if (B < 0 || H <= 0 || Sq < 0 || Sk < 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.f) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  const bool varlen = cu_seqlens_q != nullptr || cu_seqlens_k != nullptr;
  if (varlen && (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr)) return FA_ERR_INVALID_ARG;
  if (varlen && (total_q < 0 || total_k < 0)) return FA_ERR_INVALID_ARG;
  const int64_t Tq = varlen ? total_q : (int64_t)B * Sq;
  const int64_t Tk = varlen ? total_k : (int64_t)B * Sk;
  if (Tq > INT32_MAX || Tk > INT32_MAX) return FA_ERR_INVALID_ARG;
  if ((int64_t)H * D * 2 > (int64_t)1 << 38) return FA_ERR_INVALID_ARG;
  if (B == 0 || (Tq == 0 && Tk == 0)) return FA_OK;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  for (const void* p : {q, k, v, o, dout, (const void*)dq, (const void*)dk, (const void*)dv})
    if (!aligned16(p)) return FA_ERR_ALIGNMENT;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return FA_ERR_ALIGNMENT;
  const size_t need = fa_bwd_workspace_size(H, (int)Tq);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return FA_ERR_INVALID_ARG;
  if (workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FA_ERR_ALIGNMENT;
  const int64_t nq = ((int64_t)Sq + 127) / 128, nk = ((int64_t)Sk + 127) / 128;
  if ((int64_t)B * H * nq > INT32_MAX || (int64_t)B * H * nk > INT32_MAX) return FA_ERR_INVALID_ARG;

  // ---- device
  DevInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* lse2 = static_cast<float*>(workspace);
  float* delta = lse2 + (size_t)H * Tq;
  if (Tq > 0 && fa::launch_bwd_prep(o, dout, lse, lse2, delta, (int)Tq, H, D, varlen ? 1 : Sq, varlen ? 1 : 0,
                                    dtype == FA_FP16 ? 1 : 0, s) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  const CUtensorMapDataType dt = dtype == FA_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t cols = (uint64_t)H * D;
  CUtensorMap mq, mk, mv, mdo;
  if ((st = make_map(&mq, q, dt, 2, cols, (uint64_t)Tq, 64, 128)) != FA_OK) return st;
  if ((st = make_map(&mk, k, dt, 2, cols, (uint64_t)Tk, 64, 128)) != FA_OK) return st;
  if ((st = make_map(&mv, v, dt, 2, cols, (uint64_t)Tk, 64, 128)) != FA_OK) return st;
  if ((st = make_map(&mdo, dout, dt, 2, cols, (uint64_t)Tq, 64, 128)) != FA_OK) return st;
  // launches: dK and dV together, then dQ; at D = 256 (their accumulators do
  // not fit tensor memory together) dV, dK, then dQ
  const int n_dir = D == 256 ? 3 : 2;
  for (int dir = 0; dir < n_dir; ++dir) {
    fa::BwdLaunch L;
    std::memset(&L, 0, sizeof(L));
    const bool dqk = dir == n_dir - 1;
    L.part = D == 256 && !dqk ? (dir == 0 ? 2 : 1) : 0;
    L.tr1 = dqk ? mq : mk;
    L.tr2 = dqk ? mdo : mv;
    L.tt1 = dqk ? mk : mq;
    L.tt2 = dqk ? mv : mdo;
    L.p.dr1 = dqk ? dq : (L.part == 2 ? nullptr : dk);
    L.p.dr2 = dqk || L.part == 1 ? nullptr : dv;
    L.p.lse2 = lse2;
    L.p.delta = delta;
    L.p.cu_q = cu_seqlens_q;
    L.p.cu_k = cu_seqlens_k;
    L.p.B = B;
    L.p.H = H;
    L.p.Sq = Sq;
    L.p.Sk = Sk;
    L.p.total_q = (int)Tq;
    L.p.total_k = (int)Tk;
    L.p.n_rblk = (int)(dqk ? nq : nk);
    L.p.ntiles = B * H * L.p.n_rblk;
    L.p.c = (float)((double)scale * 1.4426950408889634);
    L.p.scale = scale;
    L.p.status = dev->status;
    L.D = D;
    L.kind = dtype == FA_FP16 ? fa::kF16 : fa::kBF16;
    L.causal = causal != 0;
    L.dq = dqk;
    L.p.head_group = head_group(L.causal, (int64_t)B * H, dqk ? Sk : Sq, D, 2);
    L.num_sms = dev->sms;
    L.stream = s;
    if (L.p.ntiles == 0) continue;
    SlotHold hold(dev, s);
    if ((L.p.sched = hold.sched()) == nullptr) return FA_ERR_BUSY;
    const cudaError_t e = D == 64 ? fa::launch_bwd_d64(L) : D == 128 ? fa::launch_bwd_d128(L) : fa::launch_bwd_d256(L);
    hold.launched(e == cudaSuccess);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_CUDA;
    }
  }
  return FA_OK;
}

int fa_get_device_status(void* stream, int* raw) {
  DevInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st != FA_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  int word = 0;
  const int zero = 0;
  if (cudaMemcpy(&word, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  if (raw) *raw = word;
  if (word & fa::kDevTimeout) return FA_ERR_DEVICE_TIMEOUT;
  if (word & fa::kDevBadSeqlens) return FA_ERR_DEVICE_SEQLENS;
  return FA_OK;
}

}  // extern "C"
