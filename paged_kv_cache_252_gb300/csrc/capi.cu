// C ABI of libpagedkv.so (declared in include/pagedkv.h): host-side argument
// checks, launch geometry, tensor-map encoding and kernel launches. No device
// memory is allocated here; every buffer comes from the caller.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "pagedkv.h"
#include "pkv_internal.h"

namespace {

using namespace pkv;

constexpr int kMaxDevices = 64;

struct GeomEntry {
  bool ready = false;
  DecodeGeometry geom{};
  int ctas_per_sm = 0;
  const void* fn = nullptr;
};

struct DeviceState {
  bool ready = false;
  int sm_count = 0;
  bool write_attr_done = false;
  // [kv][d==128][kernel: 0 = NTW 1, 1 = NTW 2, 2 = the 96-thread kernel for narrow units]
  GeomEntry geom[4][2][3];
  // tcgen05 kernel, [rc - 1]
  GeomEntry tc_geom[2];
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
std::atomic<uint32_t> g_call_epoch{0};
#ifdef PKV_TIMELINE
unsigned long long* g_timeline = nullptr;   // profiling build: per-CTA event buffer
int g_timeline_ctas = 0;
#endif

// Fixed cost of one unit piece on the work line, in KV blocks: the piece's
// query load, epilogue and (when split) merge take about as long as streaming
// this many blocks, so CTAs whose share starts more units get fewer blocks.
// (Compile-time overridable for tuning sweeps.)
#ifndef PKV_PIECE_COST_2B
#define PKV_PIECE_COST_2B 8
#endif
#ifndef PKV_PIECE_COST_1B
#define PKV_PIECE_COST_1B 8
#endif
#ifndef PKV_PIECE_COST_TC
#define PKV_PIECE_COST_TC 20
#endif
constexpr int kPieceCost2B = PKV_PIECE_COST_2B;   // mma.sync kernel, fp16 / bf16 cache
constexpr int kPieceCost1B = PKV_PIECE_COST_1B;   // mma.sync kernel, E5M2 / INT8 cache
constexpr int kPieceCostTc = PKV_PIECE_COST_TC;   // tcgen05 kernel (its epilogue reads O from tensor memory)
int piece_cost(bool tc, int kv) {
  if (tc) return kPieceCostTc;
  return (kv == PKV_FP8_E5M2 || kv == PKV_INT8) ? kPieceCost1B : kPieceCost2B;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int current_device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_NO_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_NO_DEVICE;
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
      cudaGetLastError();
      return PKV_ERR_NO_DEVICE;
    }
    st.sm_count = sms;
    st.ready = true;
  }
  *out = &st;
  return PKV_OK;
}

// The 96-thread kernel of its own register budget for units of at most 8 rows
// over a bf16 cache (at four CTAs per SM it beat the shared kernel at five: long
// bf16 decode 424.1 -> 412.3 us; with an fp16 cache it measured 57.1 -> 57.3 us on
// the 8B workload, and on 1-byte caches a larger budget was slower).
const void* decode_narrow_fn(int kv, int d) {
  return kv == kKvBf16 ? decode_kernel_narrow_ptr_bf16(d) : nullptr;
}

const void* decode_fn(int kv, int d, int ntw) {
  switch (kv) {
    case kKvF16: return decode_kernel_ptr_f16(d, ntw);
    case kKvBf16: return decode_kernel_ptr_bf16(d, ntw);
    case kKvE5m2: return decode_kernel_ptr_e5m2(d, ntw);
    case kKvInt8: return decode_kernel_ptr_int8(d, ntw);
    default: return nullptr;
  }
}

// Warp layout and ring depth for a unit of `rows` query rows. Consumers form a
// WR x WB grid: WR warps split the rows (8*NTW each), WB warp groups take turns
// on blocks. Each CTA has one producer thread issuing the TMA copies, and that
// thread is the limit when few CTAs share an SM, so units of at most 8 rows run
// small CTAs (2 consumer warps, ~44 KB of shared memory) five to an SM; units of
// up to 16 rows split their rows over two such warps (three CTAs per SM); wider
// units keep two larger CTAs per SM (their warps need ~168 registers).
DecodeGeometry choose_geometry(int kv, int d, int rows) {
  DecodeGeometry g{};
  const int nt = (rows + 7) / 8;
  size_t target = 110 * 1024;
  if (nt <= 1) { g.ntw = 1; g.warps_rows = 1; g.warps_blocks = 2; target = 44 * 1024; }
  else if (nt <= 2) { g.ntw = 1; g.warps_rows = 2; g.warps_blocks = 2; target = 72 * 1024; }
  else if (nt <= 4) { g.ntw = 2; g.warps_rows = 2; g.warps_blocks = 2; }
  else { g.ntw = 2; g.warps_rows = 4; g.warps_blocks = 1; }
  g.threads = (g.warps_rows * g.warps_blocks + 1) * 32;
  const size_t fixed = decode_smem_layout(kv, d, g.ntw, g.warps_rows, g.warps_blocks, 0, rows).total + 1024;
  const size_t per_stage = 2 * static_cast<size_t>(tile_bytes(kv, d)) + 16;
  long long st = target > fixed ? static_cast<long long>((target - fixed) / per_stage) : 0;
  if (st > 16) st = 16;
  // The ring depth must be a multiple of the block-stream count: then stage k is
  // only ever consumed by block-stream (k mod WB), which waits for its phases in
  // order. With any other depth a stream can reach a stage whose previous use
  // (another stream's block) has not landed yet, and the parity test of the
  // mbarrier wait cannot tell that older phase from the one it wants.
  st -= st % g.warps_blocks;
  if (st < g.warps_blocks) st = g.warps_blocks;
  if (st < 4) st = (4 + g.warps_blocks - 1) / g.warps_blocks * g.warps_blocks;
  g.stages = static_cast<int>(st);
  g.smem_bytes = decode_smem_layout(kv, d, g.ntw, g.warps_rows, g.warps_blocks, g.stages, rows).total + 1024;
  return g;
}

// Units wider than 16 rows over an E5M2 cache with head size 128 run on the
// tcgen05 kernel: one 320-thread CTA per SM holding the widened K/V chunk
// buffers, P^T, two query tiles and a ring of as many 32 KB chunk buffers
// (2..4) as fit in the 227 KB a CTA may use.
bool use_tc(int kv, int d, int rows) { return kv == kKvE5m2 && d == 128 && rows > 16; }

DecodeGeometry choose_tc_geometry(int rows) {
  DecodeGeometry g{};
  g.tc = 1;
  g.rc = rows > 32 ? 2 : 1;
  g.threads = kTcThreads;
  const size_t limit = 227 * 1024;
  int nbuf = 4;
  while (nbuf > 2 && tc_smem_layout(32 * g.rc, nbuf).total + 1024 > limit) --nbuf;
  g.stages = nbuf;
  g.smem_bytes = tc_smem_layout(32 * g.rc, nbuf).total + 1024;
  return g;
}

int get_geometry(DeviceState* st, int kv, int d, int rows, GeomEntry** out) {
  const bool tc = use_tc(kv, d, rows);
  const DecodeGeometry g0 = tc ? choose_tc_geometry(rows) : choose_geometry(kv, d, rows);
  const bool narrow = !tc && g0.warps_rows == 1 && g0.ntw == 1 && decode_narrow_fn(kv, d) != nullptr;
  GeomEntry& e = tc ? st->tc_geom[g0.rc - 1]
                    : st->geom[kv][d == 128 ? 1 : 0][narrow ? 2 : (g0.ntw == 2 ? 1 : 0)];
  // The cached entry is keyed by (kv, d, ntw); the row count also changes the
  // warp grid and the merge-buffer size, so re-derive and compare.
  if (!e.ready || e.geom.warps_rows != g0.warps_rows || e.geom.warps_blocks != g0.warps_blocks ||
      e.geom.stages != g0.stages || e.geom.smem_bytes != g0.smem_bytes || e.geom.tc != g0.tc ||
      e.geom.rc != g0.rc) {
    const void* fn = tc ? decode_tc_kernel_ptr(kv, g0.rc) : (narrow ? decode_narrow_fn(kv, d) : decode_fn(kv, d, g0.ntw));
    if (!fn) return PKV_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(g0.smem_bytes)) != cudaSuccess) {
      cudaGetLastError();
      return PKV_ERR_CUDA;
    }
    cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    cudaGetLastError();
    int nblk = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nblk, fn, g0.threads, g0.smem_bytes) !=
            cudaSuccess || nblk <= 0) {
      cudaGetLastError();
      return PKV_ERR_CUDA;
    }
    e.geom = g0;
    e.fn = fn;
    e.ctas_per_sm = nblk < kMaxCtasPerSm ? nblk : kMaxCtasPerSm;
    e.ready = true;
  }
  *out = &e;
  return PKV_OK;
}

int encode_cache_map(CUtensorMap* map, const void* base, int kv, int d, long long total_rows,
                     int half) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    cudaGetLastError();
  });
  if (!g_encode) return PKV_ERR_CUDA;
  const int rb = tile_row_bytes(kv, d);
  const int esz = kv_elem_bytes(kv);
  const CUtensorMapDataType dt = esz == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  // Every map is 2-D: [total_rows][row bytes] with a box of 16 token rows. A
  // 256-byte row (16-bit elements, head size 128) is covered by two maps, one per
  // 128-byte half (base + half*128, row stride 256), so every box is at most 128
  // bytes wide and takes the 128-byte swizzle (64-byte for 64-byte rows).
  const int box_bytes = rb > 128 ? 128 : rb;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(box_bytes / esz), static_cast<cuuint64_t>(total_rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(rb)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_bytes / esz), static_cast<cuuint32_t>(kBlockSize)};
  cuuint32_t es[2] = {1, 1};
  const char* ptr = static_cast<const char*>(base) + half * 128;
  const CUresult r = g_encode(map, dt, 2, const_cast<char*>(ptr), dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE,
                              box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

bool valid_cache(const pkv_cache_desc* c) {
  if (!c) return false;
  if (c->block_size != kBlockSize) return false;
  if (c->head_size != 64 && c->head_size != 128) return false;
  if (c->num_blocks <= 0 || c->num_kv_heads <= 0) return false;
  const long long rows = static_cast<long long>(c->num_blocks) * c->num_kv_heads * kBlockSize;
  return rows < (1ll << 31) - kBlockSize;
}

// A bijective mix of the 32-bit call number (odd multiplies and xor-shifts are
// each invertible modulo 2^32).
uint32_t call_epoch(uint32_t n) {
  n ^= n >> 16;
  n *= 0x7feb352du;
  n ^= n >> 15;
  n *= 0x846ca68bu;
  n ^= n >> 16;
  return n;
}

// Workspace layout: [per-unit piece counters, 8 bytes each, 256-aligned][partial
// slots] (decode_counter_bytes in pkv_internal.h sizes the first part).
size_t desc_bytes(long long units) { return decode_counter_bytes(units); }

// The decode grid has at most sm_count * ctas_per_sm CTAs, and a split unit's
// pieces use slots unit + cta, so units + grid slots suffice.
size_t workspace_bytes_for(long long units, int sm_count, int ctas_per_sm, int rows, int d) {
  const long long slots = units + static_cast<long long>(sm_count) * ctas_per_sm;
  return desc_bytes(units) + static_cast<size_t>(slots) * partial_slot_floats(rows, d) * sizeof(float);
}

cudaError_t launch(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, void** args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

extern "C" {

#ifdef PKV_TIMELINE
// Profiling build only (not part of the public header): decode launches after
// this call record per-CTA event times into buf ([max_ctas][8] uint64, device
// memory owned by the caller; NULL detaches). See pkv_timeline.cuh.
int pkv_timeline_attach(unsigned long long* buf, int32_t max_ctas) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_timeline = max_ctas > 0 ? buf : nullptr;
  g_timeline_ctas = buf ? max_ctas : 0;
  return PKV_OK;
}
#endif

int pkv_version(void) { return 100; }

const char* pkv_error_string(int code) {
  switch (code) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARGUMENT: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case PKV_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PKV_ERR_CUDA: return "CUDA runtime error";
    case PKV_ERR_NO_DEVICE: return "no usable CUDA device";
    case PKV_ERR_OUT_OF_BLOCKS: return "block pool exhausted";
    default: return "unknown status";
  }
}

int pkv_kv_cache_write(const void* key, const void* value, pkv_dtype src_dtype, int32_t num_tokens,
                       const int32_t* slot_mapping, void* k_cache, void* v_cache, pkv_dtype kv_dtype,
                       const pkv_cache_desc* cache, int32_t* device_status, void* stream) {
  if (num_tokens < 0 || !valid_cache(cache)) return PKV_ERR_INVALID_ARGUMENT;
  const bool pair_ok = (src_dtype == PKV_FP16 && kv_dtype == PKV_FP16) ||
                       (src_dtype == PKV_BF16 && kv_dtype == PKV_BF16) ||
                       (src_dtype == PKV_FP16 && kv_dtype == PKV_FP8_E5M2);
  if (!pair_ok) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!key || !value || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARGUMENT;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned4(slot_mapping) || (device_status && !aligned4(device_status)))
    return PKV_ERR_INVALID_ARGUMENT;

  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  if (int rc = current_device_state(&st)) return rc;

  CacheWriteArgs a{};
  a.key = static_cast<const uint4*>(key);
  a.value = static_cast<const uint4*>(value);
  a.slot_mapping = slot_mapping;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.status = device_status;
  a.num_slots = static_cast<long long>(cache->num_blocks) * kBlockSize;
  a.num_tokens = num_tokens;
  a.num_kv_heads = cache->num_kv_heads;
  a.head_size = cache->head_size;
  a.kv = static_cast<int32_t>(kv_dtype);

  const long long chunks = 2ll * num_tokens * cache->num_kv_heads * (cache->head_size / 8);
  long long blocks = (chunks + 255) / 256;
  const long long max_blocks = static_cast<long long>(st->sm_count) * 16;
  if (blocks > max_blocks) blocks = max_blocks;
  void* args[1] = {&a};
  const cudaError_t e = launch(kv_cache_write_kernel_ptr(), dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                               static_cast<cudaStream_t>(stream), args);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

size_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t q_per_seq,
                                  const pkv_cache_desc* cache) {
  if (num_seqs < 0 || num_q_heads <= 0 || q_per_seq <= 0 || !valid_cache(cache)) return 0;
  if (num_q_heads % cache->num_kv_heads != 0) return 0;
  const int rows = (num_q_heads / cache->num_kv_heads) * q_per_seq;
  if (rows > kMaxRows) return 0;
  if (cache->head_size != 64 && cache->head_size != 128) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  if (current_device_state(&st)) return 0;
  const long long units = static_cast<long long>(num_seqs) * cache->num_kv_heads;
  // The grid follows the kv dtype's occupancy; size for the largest over the
  // supported dtypes so that one workspace serves any of them.
  int ctas = 1;
  for (int kv = kKvF16; kv <= kKvInt8; ++kv) {
    GeomEntry* ge = nullptr;
    if (get_geometry(st, kv, cache->head_size, rows, &ge)) return 0;
    if (ge->ctas_per_sm > ctas) ctas = ge->ctas_per_sm;
  }
  return workspace_bytes_for(units, st->sm_count, ctas, rows, cache->head_size);
}

}  // extern "C"

namespace {

// Rows of q / out for num_seqs sequences of q_per_seq tokens (saturated; larger
// problems are refused by decode_impl's size checks).
int32_t fixed_rows(int32_t num_seqs, int32_t q_per_seq) {
  const long long r = static_cast<long long>(num_seqs) * q_per_seq;
  return r > INT32_MAX ? INT32_MAX : static_cast<int32_t>(r);
}

// Shared body of the decode entry points; cu_q_lens null means q_per_seq query
// tokens for every sequence.
int decode_impl(void* out, const void* q, const int32_t* cu_q_lens, int32_t num_q_rows,
                const unsigned long long* tree_masks, const float* scales,
                int32_t num_seqs,
                int32_t num_q_heads, int32_t q_per_seq, const void* k_cache, const void* v_cache,
                pkv_dtype kv_dtype, const pkv_cache_desc* cache, const int32_t* block_tables,
                int32_t max_blocks_per_seq, const int32_t* context_lens, float scale,
                void* workspace, size_t workspace_bytes, int32_t* device_status, void* stream) {
  if (num_seqs < 0 || num_q_heads <= 0 || q_per_seq <= 0 || max_blocks_per_seq <= 0 ||
      !valid_cache(cache))
    return PKV_ERR_INVALID_ARGUMENT;
  if (kv_dtype != PKV_FP16 && kv_dtype != PKV_BF16 && kv_dtype != PKV_FP8_E5M2 && kv_dtype != PKV_INT8)
    return PKV_ERR_UNSUPPORTED;
  if (num_q_heads % cache->num_kv_heads != 0) return PKV_ERR_INVALID_ARGUMENT;
  // An INT8 cache is read with its row scales, 16-byte aligned (a block's 16 K
  // and 16 V scales move as one 128-byte copy).
  if (kv_dtype == PKV_INT8 && (!scales || !aligned16(scales)))
    return PKV_ERR_INVALID_ARGUMENT;
  const int group = num_q_heads / cache->num_kv_heads;
  const long long rows_ll = static_cast<long long>(group) * q_per_seq;
  if (rows_ll > kMaxRows) return PKV_ERR_UNSUPPORTED;
  const int rows = static_cast<int>(rows_ll);
  if (static_cast<long long>(num_seqs) * q_per_seq * num_q_heads >= (1ll << 31))
    return PKV_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_seqs) * max_blocks_per_seq >= (1ll << 31) ||
      max_blocks_per_seq > (1 << 26))
    return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace)
    return PKV_ERR_INVALID_ARGUMENT;
  // Every row the kernels may touch lies below num_q_rows: with cu_q_lens each
  // sequence's rows are checked on the device against it; without, all
  // num_seqs * q_per_seq rows must exist.
  if (num_q_rows < 1 || (!cu_q_lens && static_cast<long long>(num_seqs) * q_per_seq > num_q_rows))
    return PKV_ERR_INVALID_ARGUMENT;
  if (cu_q_lens && !aligned4(cu_q_lens)) return PKV_ERR_INVALID_ARGUMENT;
  if (tree_masks && (reinterpret_cast<uintptr_t>(tree_masks) & 7u)) return PKV_ERR_INVALID_ARGUMENT;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(workspace) || !aligned4(block_tables) || !aligned4(context_lens) ||
      (device_status && !aligned4(device_status)))
    return PKV_ERR_INVALID_ARGUMENT;

  const int d = cache->head_size;
  const int kv = static_cast<int>(kv_dtype);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  if (int rc = current_device_state(&st)) return rc;
  const long long units = static_cast<long long>(num_seqs) * cache->num_kv_heads;
  GeomEntry* ge = nullptr;
  if (int rc = get_geometry(st, kv, d, rows, &ge)) return rc;
  const DecodeGeometry& g = ge->geom;
  if (workspace_bytes < workspace_bytes_for(units, st->sm_count, ge->ctas_per_sm, rows, d))
    return PKV_ERR_WORKSPACE_TOO_SMALL;

  const long long total_rows = static_cast<long long>(cache->num_blocks) * cache->num_kv_heads * kBlockSize;
  CUtensorMap tmk, tmv, tmk1, tmv1;
  if (int rc = encode_cache_map(&tmk, k_cache, kv, d, total_rows, 0)) return rc;
  if (int rc = encode_cache_map(&tmv, v_cache, kv, d, total_rows, 0)) return rc;
  if (tile_row_bytes(kv, d) > 128) {
    if (int rc = encode_cache_map(&tmk1, k_cache, kv, d, total_rows, 1)) return rc;
    if (int rc = encode_cache_map(&tmv1, v_cache, kv, d, total_rows, 1)) return rc;
  } else {
    tmk1 = tmk;
    tmv1 = tmv;
  }

  // One wave: every CTA resident at once; never more CTAs than blocks could exist.
  long long grid = static_cast<long long>(st->sm_count) * ge->ctas_per_sm;
  const long long max_work = units * max_blocks_per_seq;
  if (grid > max_work) grid = max_work;
  if (grid < 1) grid = 1;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeArgs a{};
  a.out = out;
  a.q = q;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.cu_q_lens = cu_q_lens;
  a.q_rows = num_q_rows;
  a.tree_masks = tree_masks;
  a.scales = kv_dtype == PKV_INT8 ? scales : nullptr;
  a.piece_counts = reinterpret_cast<unsigned long long*>(ws);
  a.partials = reinterpret_cast<float*>(ws + desc_bytes(units));
  a.status = device_status;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = cache->num_kv_heads;
  a.q_per_seq = q_per_seq;
  a.group = group;
  a.rows = rows;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = cache->num_blocks;
  a.warps_rows = g.warps_rows;
  a.warps_blocks = g.warps_blocks;
  a.stages = g.stages;
  a.slot_floats = partial_slot_floats(rows, d);
  a.scale_log2 = scale * 1.4426950408889634f;
  // Counters from an earlier call carry an older epoch and count as zero, so the
  // workspace never needs clearing. The epoch is the call number through a
  // bijective 32-bit mix, so calls never share one (within 2^32 calls) and its
  // values do not look like the small integers (lengths, block ids) a reused
  // buffer may hold; 0 and 0xFFFFFFFF are skipped (zeroed and -1-filled memory).
  uint32_t ep = 0;
  do {
    ep = call_epoch(++g_call_epoch);
  } while (ep == 0u || ep == 0xFFFFFFFFu);
  a.epoch = ep;
  a.piece_cost = piece_cost(g.tc != 0, kv_dtype);
#ifdef PKV_TIMELINE
  a.timeline = g_timeline;
  a.timeline_ctas = g_timeline_ctas;
#endif

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* dargs[5] = {&tmk, &tmv, &tmk1, &tmv1, &a};
  void* dargs_tc[3] = {&tmk, &tmv, &a};
  const cudaError_t e = launch(ge->fn, dim3(static_cast<unsigned>(grid)), dim3(g.threads), g.smem_bytes, s,
                               g.tc ? dargs_tc : dargs);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }

  return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_paged_attention_decode(void* out, const void* q, int32_t num_seqs, int32_t num_q_heads,
                               int32_t q_per_seq, const void* k_cache, const void* v_cache,
                               pkv_dtype kv_dtype, const pkv_cache_desc* cache,
                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                               const int32_t* context_lens, float scale, void* workspace,
                               size_t workspace_bytes, int32_t* device_status, void* stream) {
  return decode_impl(out, q, nullptr, fixed_rows(num_seqs, q_per_seq), nullptr, nullptr, num_seqs, num_q_heads,
                     q_per_seq, k_cache, v_cache, kv_dtype,
                     cache, block_tables, max_blocks_per_seq, context_lens, scale, workspace,
                     workspace_bytes, device_status, stream);
}

int pkv_paged_attention_decode_varlen(void* out, const void* q, const int32_t* cu_q_lens,
                                      int32_t num_q_rows, int32_t num_seqs, int32_t num_q_heads,
                                      int32_t max_q_per_seq,
                                      const void* k_cache, const void* v_cache, pkv_dtype kv_dtype,
                                      const pkv_cache_desc* cache, const int32_t* block_tables,
                                      int32_t max_blocks_per_seq, const int32_t* context_lens,
                                      float scale, void* workspace, size_t workspace_bytes,
                                      int32_t* device_status, void* stream) {
  if (num_seqs > 0 && !cu_q_lens) return PKV_ERR_INVALID_ARGUMENT;
  return decode_impl(out, q, cu_q_lens, num_q_rows, nullptr, nullptr, num_seqs, num_q_heads,
                     max_q_per_seq,
                     k_cache, v_cache,
                     kv_dtype, cache, block_tables, max_blocks_per_seq, context_lens, scale,
                     workspace, workspace_bytes, device_status, stream);
}

int pkv_paged_attention_decode_tree(void* out, const void* q, const int32_t* cu_q_lens,
                                    const uint64_t* tree_masks, int32_t num_q_rows, int32_t num_seqs,
                                    int32_t num_q_heads, int32_t max_q_per_seq,
                                    const void* k_cache, const void* v_cache, pkv_dtype kv_dtype,
                                    const pkv_cache_desc* cache, const int32_t* block_tables,
                                    int32_t max_blocks_per_seq, const int32_t* context_lens,
                                    float scale, void* workspace, size_t workspace_bytes,
                                    int32_t* device_status, void* stream) {
  if (num_seqs > 0 && !tree_masks) return PKV_ERR_INVALID_ARGUMENT;
  if (max_q_per_seq > 64) return PKV_ERR_UNSUPPORTED;
  return decode_impl(out, q, cu_q_lens, num_q_rows, reinterpret_cast<const unsigned long long*>(tree_masks), nullptr,
                     num_seqs, num_q_heads, max_q_per_seq, k_cache, v_cache, kv_dtype, cache,
                     block_tables, max_blocks_per_seq, context_lens, scale, workspace,
                     workspace_bytes, device_status, stream);
}

int pkv_paged_attention_decode_int8(void* out, const void* q, int32_t num_seqs, int32_t num_q_heads,
                                    int32_t q_per_seq, const void* k_cache, const void* v_cache,
                                    const float* scales, const pkv_cache_desc* cache,
                                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                                    const int32_t* context_lens, float scale, void* workspace,
                                    size_t workspace_bytes, int32_t* device_status, void* stream) {
  return decode_impl(out, q, nullptr, fixed_rows(num_seqs, q_per_seq), nullptr, scales, num_seqs, num_q_heads,
                     q_per_seq, k_cache,
                     v_cache, PKV_INT8, cache, block_tables, max_blocks_per_seq, context_lens, scale, workspace,
                     workspace_bytes, device_status, stream);
}

int pkv_paged_attention_decode_int8_varlen(void* out, const void* q, const int32_t* cu_q_lens,
                                           int32_t num_q_rows, int32_t num_seqs, int32_t num_q_heads,
                                           int32_t max_q_per_seq, const void* k_cache, const void* v_cache,
                                           const float* scales, const pkv_cache_desc* cache,
                                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                                           const int32_t* context_lens, float scale, void* workspace,
                                           size_t workspace_bytes, int32_t* device_status, void* stream) {
  if (num_seqs > 0 && !cu_q_lens) return PKV_ERR_INVALID_ARGUMENT;
  return decode_impl(out, q, cu_q_lens, num_q_rows, nullptr, scales, num_seqs, num_q_heads, max_q_per_seq,
                     k_cache, v_cache, PKV_INT8, cache, block_tables, max_blocks_per_seq, context_lens, scale,
                     workspace, workspace_bytes, device_status, stream);
}

int pkv_paged_attention_decode_int8_tree(void* out, const void* q, const int32_t* cu_q_lens,
                                         const uint64_t* tree_masks, int32_t num_q_rows, int32_t num_seqs,
                                         int32_t num_q_heads, int32_t max_q_per_seq, const void* k_cache,
                                         const void* v_cache, const float* scales, const pkv_cache_desc* cache,
                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                         const int32_t* context_lens, float scale, void* workspace,
                                         size_t workspace_bytes, int32_t* device_status, void* stream) {
  if (num_seqs > 0 && !tree_masks) return PKV_ERR_INVALID_ARGUMENT;
  if (max_q_per_seq > 64) return PKV_ERR_UNSUPPORTED;
  return decode_impl(out, q, cu_q_lens, num_q_rows, reinterpret_cast<const unsigned long long*>(tree_masks),
                     scales, num_seqs, num_q_heads, max_q_per_seq, k_cache, v_cache, PKV_INT8, cache, block_tables,
                     max_blocks_per_seq, context_lens, scale, workspace, workspace_bytes, device_status, stream);
}

int pkv_kv_cache_write_int8(const void* key, const void* value, int32_t num_tokens, const int32_t* slot_mapping,
                            void* k_cache, void* v_cache, float* scales,
                            const pkv_cache_desc* cache, int32_t* device_status, void* stream) {
  if (num_tokens < 0 || !valid_cache(cache)) return PKV_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return PKV_OK;
  if (!key || !value || !slot_mapping || !k_cache || !v_cache || !scales)
    return PKV_ERR_INVALID_ARGUMENT;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(scales) || !aligned4(slot_mapping) ||
      (device_status && !aligned4(device_status)))
    return PKV_ERR_INVALID_ARGUMENT;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  if (int rc = current_device_state(&st)) return rc;
  CacheWriteArgs a{};
  a.key = static_cast<const uint4*>(key);
  a.value = static_cast<const uint4*>(value);
  a.slot_mapping = slot_mapping;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.scales = scales;
  a.status = device_status;
  a.num_slots = static_cast<long long>(cache->num_blocks) * kBlockSize;
  a.num_tokens = num_tokens;
  a.num_kv_heads = cache->num_kv_heads;
  a.head_size = cache->head_size;
  a.kv = kKvInt8;
  // One warp per (token, head) row of K or V.
  const long long rows = 2ll * num_tokens * cache->num_kv_heads;
  long long blocks = (rows * 32 + 255) / 256;
  const long long max_blocks = static_cast<long long>(st->sm_count) * 16;
  if (blocks > max_blocks) blocks = max_blocks;
  void* args[1] = {&a};
  const cudaError_t e = launch(kv_cache_write_int8_kernel_ptr(), dim3(static_cast<unsigned>(blocks)), dim3(256),
                               0, static_cast<cudaStream_t>(stream), args);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

}  // extern "C"
