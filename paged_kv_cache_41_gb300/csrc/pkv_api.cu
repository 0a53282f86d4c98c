// pkv_api.cu -- the C ABI of libpkv: host-side validation, TMA descriptors,
// workspace sizing, the per-device error word and the kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <math.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "kernels/launch.h"
#include "pkv.h"

namespace {

// One error word per device; kernels get its device address.
__device__ unsigned int g_device_error;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_err_ptr[kMaxDevices] = {};

unsigned int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned int*>(p);
  }
  return g_err_ptr[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// Encoded tensor maps are pure functions of their arguments, so recently used
// ones are kept (a few hundred bytes each) and reused without re-encoding.
struct MapKey {
  CUtensorMapDataType dtype;
  cuuint32_t rank;
  void* base;
  cuuint64_t dims[5], strides[4];
  cuuint32_t box[5];
  CUtensorMapSwizzle swizzle;
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  bool used;
};
constexpr int kMapCacheSize = 64;
MapEntry g_maps[kMapCacheSize];
int g_map_next = 0;
std::mutex g_map_mu;

CUresult encode_tiled_cached(CUtensorMap* map, CUtensorMapDataType dtype, cuuint32_t rank,
                             void* base, const cuuint64_t* dims, const cuuint64_t* strides,
                             const cuuint32_t* box, CUtensorMapSwizzle swizzle) {
  MapKey k;
  memset(&k, 0, sizeof(k));
  k.dtype = dtype;
  k.rank = rank;
  k.base = base;
  for (cuuint32_t i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
    if (i + 1 < rank) k.strides[i] = strides[i];
  }
  k.swizzle = swizzle;
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int i = 0; i < kMapCacheSize; ++i)
      if (g_maps[i].used && memcmp(&g_maps[i].key, &k, sizeof(k)) == 0) {
        *map = g_maps[i].map;
        return CUDA_SUCCESS;
      }
  }
  auto enc = tensor_map_encoder();
  if (!enc) return CUDA_ERROR_NOT_INITIALIZED;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(map, dtype, rank, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) {
    std::lock_guard<std::mutex> lock(g_map_mu);
    MapEntry& e = g_maps[g_map_next];
    g_map_next = (g_map_next + 1) % kMapCacheSize;
    e.key = k;
    e.map = *map;
    e.used = true;
  }
  return r;
}

// Bytes of one element of the cache's element plane.
int elem_bytes(int dtype) { return dtype == PKV_MXFP8 ? 1 : dtype == PKV_BF16 ? 2 : 4; }
// Byte offset of an MXFP8 pool's scale plane (the element plane's size).
int64_t mx_plane_bytes(const pkv_cache_desc* c) {
  return c->num_blocks * c->block_size * c->num_kv_heads * c->head_dim;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pkv_status check_cache(const pkv_cache_desc* c) {
  if (!c) return PKV_ERR_INVALID_ARG;
  if (c->num_blocks <= 0 || c->block_size <= 0 || c->num_kv_heads <= 0 || c->head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  if (c->dtype != PKV_F32 && c->dtype != PKV_BF16 && c->dtype != PKV_MXFP8)
    return PKV_ERR_INVALID_ARG;
  return PKV_OK;
}

// Shapes the attention kernels are compiled for.
pkv_status check_attention_shape(const pkv_cache_desc* c, int32_t num_q_heads) {
  if (c->head_dim != 64 && c->head_dim != 128) return PKV_ERR_UNSUPPORTED;
  const int P = c->block_size;
  // a stage of pkv::kStageRows rows is whole blocks or a slice of one block
  const int S = pkv::kStageRows;
  if (P < 16 || P > 256 || (P <= S && S % P != 0) || (P > S && P % S != 0))
    return PKV_ERR_UNSUPPORTED;
  if (num_q_heads <= 0 || num_q_heads % c->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  const int G = num_q_heads / c->num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return PKV_ERR_UNSUPPORTED;
  // MXFP8 with more than 4 query heads per kv head: the tensor-core decode only
  if (c->dtype == PKV_MXFP8 && G > 4 &&
      !pkv::decode_tc_mx_supported(c->dtype, c->head_dim, G, c->block_size))
    return PKV_ERR_UNSUPPORTED;
  if (c->num_kv_heads > 65535 || c->num_blocks > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

// 4-D map over the pool [NB, P, Hkv, D] whose box is one kv head x `rows`
// token rows x head_dim.
pkv_status encode_cache_map(CUtensorMap* map, const pkv_cache_desc* c, const void* base,
                            int rows) {
  const cuuint64_t es = (cuuint64_t)elem_bytes(c->dtype);
  cuuint64_t dims[4] = {(cuuint64_t)c->head_dim, (cuuint64_t)c->num_kv_heads,
                        (cuuint64_t)c->block_size, (cuuint64_t)c->num_blocks};
  cuuint64_t strides[3] = {dims[0] * es, dims[0] * dims[1] * es, dims[0] * dims[1] * dims[2] * es};
  cuuint32_t box[4] = {(cuuint32_t)c->head_dim, 1, (cuuint32_t)rows, 1};
  const CUtensorMapDataType dt = c->dtype == PKV_BF16    ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                : c->dtype == PKV_MXFP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUresult r = encode_tiled_cached(map, dt,
                                   4, const_cast<void*>(base), dims, strides, box,
                                   CU_TENSOR_MAP_SWIZZLE_NONE);
  if (r == CUDA_ERROR_NOT_INITIALIZED) return PKV_ERR_CUDA;
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_UNSUPPORTED;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

// Whether the decode runs on the tensor cores (eight query heads per kv
// head) or on the CUDA cores, and the rows of one stage of its work list.
// Eight query heads per kv head run on the tensor cores (bf16, and MXFP8
// through the widening kernel); fewer on the CUDA cores, which for MXFP8
// pools measure faster than widening to bf16 in shared memory (266 vs
// 377 us for the Llama-shaped layer: the widening, not HBM, bounds the
// tensor-core kernel).
bool use_tc_decode(const pkv_cache_desc* c, int group) {
  return pkv::decode_tc_supported(c->dtype, c->head_dim, group, c->block_size) ||
         pkv::decode_tc_mx_supported(c->dtype, c->head_dim, group, c->block_size);
}

int decode_stage_rows(const pkv_cache_desc* c, int group) {
  return use_tc_decode(c, group) ? pkv::decode_tc_rows() : pkv::kStageRows;
}

// Stages in the decode work list at most: every (sequence, kv head) at
// max_blocks * P rows.
int64_t max_decode_stages(const pkv_cache_desc* c, int group, int32_t num_seqs,
                          int32_t max_blocks) {
  const int64_t rows = (int64_t)max_blocks * c->block_size;
  const int sr = decode_stage_rows(c, group);
  return (int64_t)num_seqs * c->num_kv_heads * ((rows + sr - 1) / sr);
}

// CTAs of the persistent decode kernel: one wave of resident CTAs (fewer
// when there are fewer stages); partition_size > 0 adds CTAs until none
// streams more than partition_size rows (at least one stage each).
int64_t decode_ctas(const pkv_cache_desc* c, int32_t num_seqs, int32_t num_q_heads,
                    int32_t max_blocks, int32_t partition_size) {
  const int G = num_q_heads / c->num_kv_heads;
  const bool tc = use_tc_decode(c, G);
  int64_t resident = !tc ? pkv::decode_resident_ctas(c->dtype, c->head_dim, G)
                     : c->dtype == PKV_MXFP8 ? pkv::decode_tc_mx_resident_ctas()
                                             : pkv::decode_tc_resident_ctas();
  if (resident <= 0) resident = (tc ? 1LL : 4LL) * sm_count();
  const int64_t smax = max_decode_stages(c, G, num_seqs, max_blocks);
  int64_t C = resident < smax ? resident : smax;
  if (partition_size > 0) {
    int64_t cap = partition_size / decode_stage_rows(c, G);
    if (cap < 1) cap = 1;
    const int64_t need = (smax + cap - 1) / cap;
    if (need > C) C = need;
  }
  // work units per CTA fit an int: at most 2 per stage plus 3 per piece,
  // 5 per stage when every segment is one stage
  const int64_t fit = (5 * smax + (1LL << 30) - 1) >> 30;
  if (fit > C) C = fit;
  return C < 1 ? 1 : C;
}

pkv_status encode_q_map_sw128(CUtensorMap* map, const void* q, int32_t num_seqs,
                              int32_t num_q_heads, int32_t head_dim, int group, int rpb);
pkv_status encode_cache_map_rg(CUtensorMap* map, const pkv_cache_desc* c, const void* base,
                               int rows);

// Encode the maps and launch the decode (partial kernel + reduction) on the
// path use_tc_decode picks.
pkv_status launch_decode(const pkv_cache_desc* cache, int G, const void* q, const void* k_cache,
                         const void* v_cache, const pkv::DecodeArgs& args, cudaStream_t stream,
                         int32_t q_seqs = 0) {
  pkv_status st;
  CUtensorMap tmk, tmv;
  cudaError_t e;
  pkv::DecodeArgs a = args;
  // Work units of the split (kernels/plan.cuh).  A piece's fixed cost (its
  // q, the merge of the four warps and its record) is about one and a half
  // 32-row stages of the CUDA-core decode, so there a piece weighs three
  // units and a stage two.  Where segments are short this decides the
  // balance; where they are long it costs nothing.  Measured against equal
  // stage shares: churn trace 4,960 -> 5,080 GB/s, shared-prefix call
  // 69 -> 65.5 us, prefix-tree call 77 -> 72 us, the long-context decode
  // unchanged; a piece worth 1/4, 1/3, 1/2, 3/4, 1 or 2 stages measured no
  // better overall.  The tensor-core decode's 128-row stages dwarf a piece.
  const bool tc = use_tc_decode(cache, G);
  if (cache->dtype == PKV_MXFP8) {  // the scale planes follow the element planes
    a.k_scales = static_cast<const uint8_t*>(k_cache) + mx_plane_bytes(cache);
    a.v_scales = static_cast<const uint8_t*>(v_cache) + mx_plane_bytes(cache);
  }
  a.stage_units = tc ? 1 : 2;
  a.piece_units = tc ? 0 : 3;
  if (tc) {
    const int rows = cache->block_size < pkv::decode_tc_rows() ? cache->block_size
                                                               : pkv::decode_tc_rows();
    CUtensorMap tmq;
    if (cache->dtype == PKV_MXFP8) {  // 128-byte E4M3 rows, widened in the kernel
      if ((st = encode_cache_map(&tmk, cache, k_cache, rows)) != PKV_OK) return st;
      if ((st = encode_cache_map(&tmv, cache, v_cache, rows)) != PKV_OK) return st;
      if ((st = encode_q_map_sw128(&tmq, q, q_seqs > 0 ? q_seqs : a.num_seqs, a.num_q_heads,
                                   cache->head_dim, G, 1)) != PKV_OK)
        return st;
      e = pkv::launch_paged_decode_tc_mx(G, tmk, tmv, tmq, a, stream);
      return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
    }
    if ((st = encode_cache_map_rg(&tmk, cache, k_cache, rows)) != PKV_OK) return st;
    if ((st = encode_cache_map_rg(&tmv, cache, v_cache, rows)) != PKV_OK) return st;
    if ((st = encode_q_map_sw128(&tmq, q, q_seqs > 0 ? q_seqs : a.num_seqs, a.num_q_heads,
                                 cache->head_dim, G, 1)) !=
        PKV_OK)
      return st;
    e = pkv::launch_paged_decode_tc(tmk, tmv, tmq, a, stream);
  } else {
    const int rows = pkv::box_rows_for(cache->block_size);
    if ((st = encode_cache_map(&tmk, cache, k_cache, rows)) != PKV_OK) return st;
    if ((st = encode_cache_map(&tmv, cache, v_cache, rows)) != PKV_OK) return st;
    e = pkv::launch_paged_decode(cache->dtype, cache->head_dim, G, tmk, tmv, a, stream);
  }
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// Decode workspace: stage prefix [B + 1] int64, piece LSEs [2C, G] and piece
// outputs [2C, G, D] fp32, each 256-byte aligned.
struct DecodeWorkspace {
  size_t pre_off, lse_off, o_off, total;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

DecodeWorkspace decode_workspace(int64_t num_seqs, int64_t ctas, int64_t group, int64_t head_dim) {
  DecodeWorkspace w;
  w.pre_off = 0;
  w.lse_off = align256((size_t)(num_seqs + 1) * 8);
  w.o_off = w.lse_off + align256((size_t)(2 * ctas * group) * 4);
  w.total = w.o_off + align256((size_t)(2 * ctas * group * head_dim) * 4);
  return w;
}

// Point the decode arguments' plan and piece records into a workspace.
void bind_decode_workspace(pkv::DecodeArgs* a, void* base, const DecodeWorkspace& w) {
  unsigned char* b = static_cast<unsigned char*>(base);
  a->plan_pre = reinterpret_cast<int64_t*>(b + w.pre_off);
  a->rec_lse = reinterpret_cast<float*>(b + w.lse_off);
  a->rec_o = reinterpret_cast<float*>(b + w.o_off);
}


// 3-D map over q [B, Hq, D] (bf16) with 128-byte swizzle; box = 64 columns x
// G heads x rpb requests.
pkv_status encode_q_map_sw128(CUtensorMap* map, const void* q, int32_t num_seqs, int32_t num_q_heads,
                              int32_t head_dim, int group, int rpb) {
  cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_q_heads, (cuuint64_t)num_seqs};
  cuuint64_t strides[2] = {dims[0] * 2, dims[0] * dims[1] * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)rpb};
  CUresult r = encode_tiled_cached(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q),
                                   dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  if (r == CUDA_ERROR_NOT_INITIALIZED) return PKV_ERR_CUDA;
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_UNSUPPORTED;
}

// Row-group map over a bf16 pool (kernels/launch.h): 5-D (64 columns, 8
// rows, D / 64 halves, Hkv, NB * P / 8 row groups) with 128-byte swizzle;
// box = `rows` token rows (a multiple of 8) of one head, every half.
pkv_status encode_cache_map_rg(CUtensorMap* map, const pkv_cache_desc* c, const void* base,
                               int rows) {
  const cuuint64_t row_bytes = (cuuint64_t)c->num_kv_heads * c->head_dim * 2;
  const int rg = pkv::kRowGroup;
  // the kernels address row groups with int32 coordinates
  if ((int64_t)c->num_blocks * (c->block_size / rg) > INT32_MAX || c->block_size % rg != 0)
    return PKV_ERR_UNSUPPORTED;
  cuuint64_t dims[5] = {64, (cuuint64_t)rg, (cuuint64_t)(c->head_dim / 64),
                        (cuuint64_t)c->num_kv_heads,
                        (cuuint64_t)c->num_blocks * (cuuint64_t)(c->block_size / rg)};
  cuuint64_t strides[4] = {row_bytes, 128, (cuuint64_t)c->head_dim * 2, row_bytes * rg};
  cuuint32_t box[5] = {64, (cuuint32_t)rg, (cuuint32_t)(c->head_dim / 64), 1,
                       (cuuint32_t)(rows / rg)};
  CUresult r = encode_tiled_cached(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base),
                                   dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  if (r == CUDA_ERROR_NOT_INITIALIZED) return PKV_ERR_CUDA;
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_UNSUPPORTED;
}


// Prefix K/V maps: one box is one block (or 128 rows of a larger one).
pkv_status encode_prefix_maps(CUtensorMap* tmk, CUtensorMap* tmv, const pkv_cache_desc* c,
                              const void* k_cache, const void* v_cache) {
  const int rows = c->block_size < pkv::kPrefixKeys ? c->block_size : pkv::kPrefixKeys;
  pkv_status st = encode_cache_map_rg(tmk, c, k_cache, rows);
  return st != PKV_OK ? st : encode_cache_map_rg(tmv, c, v_cache, rows);
}

// Prefix state outputs [B, Hq, parts_stride, D] fp32 as the 5-D tensor
// (D, parts_stride, G, Hkv, B); one store box is 32 columns (128 bytes, the
// swizzle span) of one split for the 128 rows (128 / G requests x G heads)
// of a query tile.
pkv_status encode_prefix_out_map(CUtensorMap* map, float* part_o, int32_t num_seqs,
                                 int32_t num_kv_heads, int group, int32_t parts_stride,
                                 int32_t head_dim) {
  const cuuint64_t row = (cuuint64_t)head_dim * 4;
  cuuint64_t dims[5] = {(cuuint64_t)head_dim, (cuuint64_t)parts_stride, (cuuint64_t)group,
                        (cuuint64_t)num_kv_heads, (cuuint64_t)num_seqs};
  cuuint64_t strides[4] = {row, row * parts_stride, row * parts_stride * group,
                           row * parts_stride * group * num_kv_heads};
  cuuint32_t box[5] = {32, 1, (cuuint32_t)group, 1, (cuuint32_t)(pkv::kPrefixRows / group)};
  CUresult r = encode_tiled_cached(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, part_o, dims, strides,
                                   box, CU_TENSOR_MAP_SWIZZLE_128B);
  if (r == CUDA_ERROR_NOT_INITIALIZED) return PKV_ERR_CUDA;
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_UNSUPPORTED;
}

// Keys per prefix split: whole 128-key tiles, spread so that (split x pair of
// query tiles x kv head) CTAs cover the SMs about once.
int32_t prefix_split_len(const pkv_cache_desc* c, int32_t num_seqs, int32_t num_q_heads,
                         int32_t prefix_len) {
  const int G = num_q_heads / c->num_kv_heads;
  const int64_t m_tiles = ((int64_t)num_seqs * G + pkv::kPrefixRows - 1) / pkv::kPrefixRows;
  const int64_t pairs = (m_tiles + 1) / 2 * c->num_kv_heads;
  const int64_t tiles = (prefix_len + pkv::kPrefixKeys - 1) / pkv::kPrefixKeys;
  int64_t splits = (sm_count() + pairs / 2) / pairs;
  if (splits < 1) splits = 1;
  if (splits > tiles) splits = tiles;
  const int64_t per = (tiles + splits - 1) / splits;
  return (int32_t)(per * pkv::kPrefixKeys);
}

// Shapes the shared-prefix path is compiled for (bf16 tensor cores).
pkv_status check_prefix_shape(const pkv_cache_desc* c, int32_t num_q_heads, int32_t prefix_len) {
  pkv_status st = check_attention_shape(c, num_q_heads);
  if (st != PKV_OK) return st;
  if (c->dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
  const int P = c->block_size;
  if (pkv::kPrefixKeys % P != 0 && P % pkv::kPrefixKeys != 0) return PKV_ERR_UNSUPPORTED;
  if (prefix_len < 0 || prefix_len % P != 0) return PKV_ERR_INVALID_ARG;
  return PKV_OK;
}

// Shared-prefix states: [B, Hq, stride] x (D floats of output + 1 LSE).
size_t states_bytes(int64_t rows, int64_t stride, int64_t head_dim) {
  return align256((size_t)(rows * stride * head_dim) * 4) + align256((size_t)(rows * stride) * 4);
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_DEVICE: return "device-side error reported by a kernel";
    case PKV_ERR_CAPACITY: return "request needs more scratch than the library's fixed device array";
  }
  return "unknown status";
}

pkv_status pkv_kv_append(const pkv_cache_desc* cache, void* k_cache, void* v_cache,
                         const void* k, const void* v, const int64_t* slot_mapping,
                         int64_t num_tokens, void* stream) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k_cache || !v_cache || !k || !v || !slot_mapping) return PKV_ERR_INVALID_ARG;
  const int64_t row_bytes = (int64_t)cache->num_kv_heads * cache->head_dim * elem_bytes(cache->dtype);
  if (row_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k) || !aligned16(v))
    return PKV_ERR_INVALID_ARG;
  if ((num_tokens * cache->num_kv_heads + 7) / 8 > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  unsigned int* err = device_error_word();
  if (!err) return PKV_ERR_CUDA;
  cudaError_t e;
  if (cache->dtype == PKV_MXFP8) {  // quantize bf16 rows into the two planes
    if (cache->head_dim != 64 && cache->head_dim != 128) return PKV_ERR_UNSUPPORTED;
    e = pkv::launch_kv_append_mxfp8(k_cache, v_cache, k, v, slot_mapping, num_tokens,
                                    cache->num_kv_heads, cache->head_dim, cache->block_size,
                                    cache->num_blocks * cache->block_size, mx_plane_bytes(cache),
                                    err, as_stream(stream));
  } else {
    e = pkv::launch_kv_append(k_cache, v_cache, k, v, slot_mapping, num_tokens,
                              cache->num_blocks * cache->block_size, row_bytes, err,
                              as_stream(stream));
  }
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_kv_block_copy(const pkv_cache_desc* cache, void* k_cache, void* v_cache,
                             const int64_t* src_dst_pairs, int64_t num_pairs, void* stream) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (num_pairs < 0) return PKV_ERR_INVALID_ARG;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !src_dst_pairs) return PKV_ERR_INVALID_ARG;
  const int64_t block_bytes = (int64_t)cache->block_size * cache->num_kv_heads * cache->head_dim *
                              elem_bytes(cache->dtype);
  if (block_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
  if (cache->dtype == PKV_MXFP8 && (cache->head_dim % 32 != 0 || (block_bytes / 32) % 16 != 0))
    return PKV_ERR_UNSUPPORTED;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_INVALID_ARG;
  if (num_pairs > INT32_MAX || block_bytes / 16 / 1024 + 1 > 65535) return PKV_ERR_UNSUPPORTED;
  unsigned int* err = device_error_word();
  if (!err) return PKV_ERR_CUDA;
  cudaError_t e = pkv::launch_kv_block_copy(k_cache, v_cache, src_dst_pairs, num_pairs,
                                            cache->num_blocks, block_bytes, err, as_stream(stream));
  if (e == cudaSuccess && cache->dtype == PKV_MXFP8) {
    // the scale plane holds a block's scales contiguously too: copy them alike
    const int64_t plane = mx_plane_bytes(cache);
    e = pkv::launch_kv_block_copy(static_cast<unsigned char*>(k_cache) + plane,
                                  static_cast<unsigned char*>(v_cache) + plane, src_dst_pairs,
                                  num_pairs, cache->num_blocks, block_bytes / 32, err,
                                  as_stream(stream));
  }
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_expand_block_tables(const int32_t* tables, int32_t num_seqs, int32_t max_blocks,
                                   int32_t alloc_block_size, int32_t kernel_block_size,
                                   int32_t* out, void* stream) {
  if (num_seqs < 0 || max_blocks < 0 || alloc_block_size <= 0 || kernel_block_size <= 0 ||
      alloc_block_size % kernel_block_size != 0)
    return PKV_ERR_INVALID_ARG;
  const int64_t n_in = (int64_t)num_seqs * max_blocks;
  if (n_in == 0) return PKV_OK;
  if (!tables || !out) return PKV_ERR_INVALID_ARG;
  const int32_t q = alloc_block_size / kernel_block_size;
  if ((int64_t)max_blocks * q > INT32_MAX || n_in * q > ((int64_t)1 << 40))
    return PKV_ERR_UNSUPPORTED;
  unsigned int* err = device_error_word();
  if (!err) return PKV_ERR_CUDA;
  cudaError_t e = pkv::launch_expand_block_tables(tables, n_in, q, out, err, as_stream(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int32_t pkv_decode_num_ctas(const pkv_cache_desc* cache, int32_t num_seqs, int32_t num_q_heads,
                            int32_t max_blocks_per_seq, int32_t partition_size) {
  if (check_cache(cache) != PKV_OK || max_blocks_per_seq <= 0 || num_seqs <= 0 ||
      partition_size < 0 || check_attention_shape(cache, num_q_heads) != PKV_OK ||
      partition_size % cache->block_size != 0)
    return 0;
  const int64_t C = decode_ctas(cache, num_seqs, num_q_heads, max_blocks_per_seq, partition_size);
  return C > INT32_MAX ? 0 : (int32_t)C;
}

size_t pkv_decode_workspace_bytes(const pkv_cache_desc* cache, int32_t num_seqs,
                                  int32_t num_q_heads, int32_t max_blocks_per_seq,
                                  int32_t partition_size) {
  if (check_cache(cache) != PKV_OK || num_seqs <= 0 || num_q_heads <= 0 ||
      max_blocks_per_seq <= 0 || partition_size < 0 ||
      check_attention_shape(cache, num_q_heads) != PKV_OK ||
      partition_size % cache->block_size != 0)
    return 0;
  const int64_t C = decode_ctas(cache, num_seqs, num_q_heads, max_blocks_per_seq, partition_size);
  return decode_workspace(num_seqs, C, num_q_heads / cache->num_kv_heads, cache->head_dim).total;
}

pkv_status pkv_paged_attention_decode(const pkv_cache_desc* cache, void* out, float* lse,
                                      const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* seq_lens, int32_t num_seqs,
                                      int32_t num_q_heads, float scale, int32_t partition_size,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || max_blocks_per_seq <= 0 || partition_size < 0 || !isfinite(scale))
    return PKV_ERR_INVALID_ARG;
  if ((st = check_attention_shape(cache, num_q_heads)) != PKV_OK) return st;
  if (num_seqs == 0) return PKV_OK;
  if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  if (partition_size % cache->block_size != 0) return PKV_ERR_INVALID_ARG;
  const int G = num_q_heads / cache->num_kv_heads;
  const int64_t C = decode_ctas(cache, num_seqs, num_q_heads, max_blocks_per_seq, partition_size);
  if (C > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  const DecodeWorkspace w = decode_workspace(num_seqs, C, G, cache->head_dim);
  if (workspace_bytes < w.total || !workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PKV_ERR_INVALID_ARG;

  unsigned int* err = device_error_word();
  if (!err) return PKV_ERR_CUDA;

  pkv::DecodeArgs a{};
  a.q = q;
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.out = out;
  a.lse_out = lse;
  a.err = err;
  bind_decode_workspace(&a, workspace, w);
  a.num_blocks = cache->num_blocks;
  a.max_blocks = max_blocks_per_seq;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = cache->num_kv_heads;
  a.block_size = cache->block_size;
  a.num_ctas = (int32_t)C;
  a.num_stages = pkv::decode_num_stages(cache->head_dim, elem_bytes(cache->dtype));
  a.qscale = scale * 1.4426950408889634f;
  // The length scan runs under the preceding kernel's tail where that kernel
  // lets its dependents start early (kv_append: it writes rows, never lengths)
  a.plan_before_wait = 1;
  return launch_decode(cache, G, q, k_cache, v_cache, a, as_stream(stream));
}

// Shared-prefix workspace: prefix states plus the suffix's whole-segment
// state ([B, Hq, prefix splits + 1] x (D + 1) fp32), then the suffix
// decode's plan and piece records.
struct SharedWorkspace {
  int32_t split_len, prefix_parts;
  int64_t ctas;
  size_t st_lse_off, dec_off, total;
  DecodeWorkspace dec;
};

SharedWorkspace shared_workspace(const pkv_cache_desc* c, int32_t num_seqs, int32_t num_q_heads,
                                 int32_t prefix_len, int32_t max_suffix_blocks,
                                 int32_t partition_size) {
  SharedWorkspace w{};
  if (prefix_len > 0) {
    w.split_len = prefix_split_len(c, num_seqs, num_q_heads, prefix_len);
    w.prefix_parts = (prefix_len + w.split_len - 1) / w.split_len;
  }
  const int64_t rows = (int64_t)num_seqs * num_q_heads, stride = w.prefix_parts + 1;
  w.st_lse_off = align256((size_t)(rows * stride * c->head_dim) * 4);
  w.dec_off = states_bytes(rows, stride, c->head_dim);
  w.ctas = decode_ctas(c, num_seqs, num_q_heads, max_suffix_blocks, partition_size);
  w.dec = decode_workspace(num_seqs, w.ctas, num_q_heads / c->num_kv_heads, c->head_dim);
  w.total = w.dec_off + w.dec.total;
  return w;
}

size_t pkv_shared_prefix_workspace_bytes(const pkv_cache_desc* cache, int32_t num_seqs,
                                         int32_t num_q_heads, int32_t prefix_len,
                                         int32_t max_suffix_blocks, int32_t partition_size) {
  if (check_cache(cache) != PKV_OK || num_seqs <= 0 || num_q_heads <= 0 || max_suffix_blocks <= 0 ||
      partition_size < 0 || check_prefix_shape(cache, num_q_heads, prefix_len) != PKV_OK ||
      partition_size % cache->block_size != 0)
    return 0;
  return shared_workspace(cache, num_seqs, num_q_heads, prefix_len, max_suffix_blocks,
                          partition_size)
      .total;
}

pkv_status pkv_shared_prefix_attention(
    const pkv_cache_desc* cache, void* out, float* lse, const void* q, const void* k_cache,
    const void* v_cache, const int32_t* prefix_block_ids, int32_t prefix_len,
    const int32_t* suffix_block_tables, int32_t max_suffix_blocks, const int32_t* suffix_lens,
    int32_t num_seqs, int32_t num_q_heads, float scale, int32_t partition_size, void* workspace,
    size_t workspace_bytes, void* stream) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || max_suffix_blocks <= 0 || partition_size < 0 || !isfinite(scale))
    return PKV_ERR_INVALID_ARG;
  if ((st = check_prefix_shape(cache, num_q_heads, prefix_len)) != PKV_OK) return st;
  if (num_seqs == 0) return PKV_OK;
  if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
  if (!out || !q || !k_cache || !v_cache || !suffix_block_tables || !suffix_lens ||
      (prefix_len > 0 && !prefix_block_ids))
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  if (partition_size % cache->block_size != 0) return PKV_ERR_INVALID_ARG;
  const SharedWorkspace w = shared_workspace(cache, num_seqs, num_q_heads, prefix_len,
                                             max_suffix_blocks, partition_size);
  if (w.ctas > INT32_MAX || w.prefix_parts >= INT32_MAX) return PKV_ERR_UNSUPPORTED;
  if (workspace_bytes < w.total || !workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PKV_ERR_INVALID_ARG;
  const int G = num_q_heads / cache->num_kv_heads;
  unsigned int* err = device_error_word();
  if (!err) return PKV_ERR_CUDA;
  unsigned char* base = static_cast<unsigned char*>(workspace);
  float* st_o = reinterpret_cast<float*>(base);
  float* st_lse = reinterpret_cast<float*>(base + w.st_lse_off);
  const int32_t stride = w.prefix_parts + 1;
  const float qscale = scale * 1.4426950408889634f;
  cudaStream_t s = as_stream(stream);

  if (w.prefix_parts > 0) {
    CUtensorMap tmq;
    if ((st = encode_q_map_sw128(&tmq, q, num_seqs, num_q_heads, cache->head_dim, G,
                                 pkv::kPrefixRows / G)) != PKV_OK)
      return st;
    pkv::PrefixArgs pa{};
    pa.prefix_block_ids = prefix_block_ids;
    pa.part_o = st_o;
    pa.part_lse = st_lse;
    pa.err = err;
    pa.num_blocks = cache->num_blocks;
    pa.num_seqs = num_seqs;
    pa.num_q_heads = num_q_heads;
    pa.num_kv_heads = cache->num_kv_heads;
    pa.block_size = cache->block_size;
    pa.prefix_len = prefix_len;
    pa.split_len = w.split_len;
    pa.parts_stride = stride;
    pa.qscale = qscale;
    pa.lse_scale = 1.f;
    CUtensorMap ptk, ptv, pto;
    if ((st = encode_prefix_maps(&ptk, &ptv, cache, k_cache, v_cache)) != PKV_OK) return st;
    if ((st = encode_prefix_out_map(&pto, st_o, num_seqs, cache->num_kv_heads, G, stride,
                                    cache->head_dim)) != PKV_OK)
      return st;
    if (pkv::launch_prefix_attention(cache->head_dim, G, w.prefix_parts, tmq, ptk, ptv, pto, pa,
                                     s) != cudaSuccess)
      return PKV_ERR_CUDA;
  }

  pkv::DecodeArgs a{};
  a.q = q;
  a.block_tables = suffix_block_tables;
  a.seq_lens = suffix_lens;
  a.out = out;
  a.lse_out = lse;
  a.err = err;
  bind_decode_workspace(&a, base + w.dec_off, w.dec);
  a.st_o = st_o;
  a.st_lse = st_lse;
  a.st_stride = stride;
  a.st_slot = w.prefix_parts;
  a.num_blocks = cache->num_blocks;
  a.max_blocks = max_suffix_blocks;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = cache->num_kv_heads;
  a.block_size = cache->block_size;
  a.num_ctas = (int32_t)w.ctas;
  a.num_stages = pkv::decode_num_stages(cache->head_dim, elem_bytes(cache->dtype));
  a.qscale = qscale;
  a.plan_before_wait = w.prefix_parts > 0;  // right after the prefix kernel
  return launch_decode(cache, G, q, k_cache, v_cache, a, s);
}

int32_t pkv_prefix_split_len(const pkv_cache_desc* cache, int32_t num_seqs, int32_t num_q_heads,
                             int32_t prefix_len) {
  if (check_cache(cache) != PKV_OK || num_seqs <= 0 || prefix_len <= 0 ||
      check_prefix_shape(cache, num_q_heads, prefix_len) != PKV_OK)
    return 0;
  return prefix_split_len(cache, num_seqs, num_q_heads, prefix_len);
}

pkv_status pkv_prefix_attention_states(const pkv_cache_desc* cache, float* states_o,
                                       float* states_lse, const void* q, const void* k_cache,
                                       const void* v_cache, const int32_t* prefix_block_ids,
                                       int32_t prefix_len, int32_t split_len, int32_t num_seqs,
                                       int32_t num_q_heads, float scale, void* stream) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || prefix_len <= 0 || split_len <= 0 || split_len % pkv::kPrefixKeys != 0 ||
      !isfinite(scale))
    return PKV_ERR_INVALID_ARG;
  if ((st = check_prefix_shape(cache, num_q_heads, prefix_len)) != PKV_OK) return st;
  if (num_seqs == 0) return PKV_OK;
  if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
  if (!states_o || !states_lse || !q || !k_cache || !v_cache || !prefix_block_ids)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(states_o) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  const int64_t splits = ((int64_t)prefix_len + split_len - 1) / split_len;
  if (splits > 65535) return PKV_ERR_UNSUPPORTED;
  if (pkv::prefix_smem_bytes(cache->head_dim, split_len, cache->block_size) > 227 * 1024)
    return PKV_ERR_UNSUPPORTED;
  const int G = num_q_heads / cache->num_kv_heads;
  unsigned int* err = device_error_word();
  if (!err) return PKV_ERR_CUDA;
  CUtensorMap tmq;
  if ((st = encode_q_map_sw128(&tmq, q, num_seqs, num_q_heads, cache->head_dim, G,
                               pkv::kPrefixRows / G)) != PKV_OK)
    return st;
  pkv::PrefixArgs pa{};
  pa.prefix_block_ids = prefix_block_ids;
  pa.part_o = states_o;
  pa.part_lse = states_lse;
  pa.err = err;
  pa.num_blocks = cache->num_blocks;
  pa.num_seqs = num_seqs;
  pa.num_q_heads = num_q_heads;
  pa.num_kv_heads = cache->num_kv_heads;
  pa.block_size = cache->block_size;
  pa.prefix_len = prefix_len;
  pa.split_len = split_len;
  pa.parts_stride = (int32_t)splits;
  pa.qscale = scale * 1.4426950408889634f;
  pa.lse_scale = 0.6931471805599453f;
  CUtensorMap ptk, ptv, pto;
  if ((st = encode_prefix_maps(&ptk, &ptv, cache, k_cache, v_cache)) != PKV_OK) return st;
  if ((st = encode_prefix_out_map(&pto, states_o, num_seqs, cache->num_kv_heads, G, (int32_t)splits,
                                  cache->head_dim)) != PKV_OK)
    return st;
  cudaError_t e = pkv::launch_prefix_attention(cache->head_dim, G, (int)splits, tmq, ptk, ptv, pto,
                                               pa, as_stream(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_get_device_error(int32_t* code_out, void* stream) {
  if (!code_out) return PKV_ERR_INVALID_ARG;
  unsigned int* err = device_error_word();
  if (!err) return PKV_ERR_CUDA;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return PKV_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return PKV_ERR_CUDA;
  const unsigned int zero = 0;
  if (cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return PKV_ERR_CUDA;
  *code_out = (int32_t)v;
  return v ? PKV_ERR_DEVICE : PKV_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free decode.  Same computation as pkv_paged_attention_decode, but
// the split-K partial states live in a fixed array that the library itself
// owns in device global memory, so the caller passes no workspace and nothing
// here allocates.
// ---------------------------------------------------------------------------
}  // extern "C"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[PKV_STATIC_SCRATCH_BYTES];

std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device.  Looked up once
// per device (with that device current) and cached; NULL if the lookup fails.
void* static_scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return nullptr;
    g_static_ptr[dev] = p;
  }
  return g_static_ptr[dev];
}

}  // namespace

extern "C" {

pkv_status pkv_paged_attention_decode_static(
    const pkv_cache_desc* cache, void* out, float* lse, const void* q, const void* k_cache,
    const void* v_cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads, float scale,
    int32_t partition_size, void* stream) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || max_blocks_per_seq <= 0 || partition_size < 0 || !isfinite(scale))
    return PKV_ERR_INVALID_ARG;
  if ((st = check_attention_shape(cache, num_q_heads)) != PKV_OK) return st;
  if (num_seqs == 0) return PKV_OK;
  if (partition_size % cache->block_size != 0) return PKV_ERR_INVALID_ARG;
  const size_t need = pkv_decode_workspace_bytes(cache, num_seqs, num_q_heads, max_blocks_per_seq,
                                                 partition_size);
  if (need == 0) return PKV_ERR_INVALID_ARG;
  if (need > (size_t)PKV_STATIC_SCRATCH_BYTES) return PKV_ERR_CAPACITY;
  void* scratch = static_scratch_address();
  if (!scratch) return PKV_ERR_CUDA;
  return pkv_paged_attention_decode(cache, out, lse, q, k_cache, v_cache, block_tables,
                                    max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, scale,
                                    partition_size, scratch, need, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Attention over a prefix tree ("M5.3 - KV Memory Layout and Exact Reuse",
// 0x0BB-0x0BE).  The host plans the snapshot into one byte blob: a header,
// then 256-byte aligned sections
//   items    PrefixItem [n_items]       chunk-first work (tensor cores)
//   cf_ids   int32 [..]                 block ids of the chunk-first chunks
//   ptab     int32 [n_pseudo, pmax]     block table of each sequence-first
//                                       (sequence, chunk) segment, -1 padded
//   plen     int32 [n_pseudo]           its rows
//   pq       int32 [n_pseudo]           its sequence (q row)
//   seq_ptr  int32 [B + 1]              CSR over states, per sequence
//   states   int64 [n_states][2]        (base, head stride): the state of
//                                       query head h is base + h * stride
// and sizes the device workspace: chunk-first states [cf_rows, Hq, s_max]
// followed by segment states [n_pseudo, Hq] (O fp32 [.., D] in one array,
// LSE base 2 in another), then the paged decode's plan and piece records.
// ---------------------------------------------------------------------------
namespace {

constexpr uint32_t kTreePlanMagic = 0x54564B50u;  // bytes "PKVT"
constexpr uint32_t kTreePlanVersion = 1;
constexpr size_t kTreePlanHeader = 256;

struct TreePlanHeader {
  uint32_t magic, version;
  int64_t num_blocks;
  int32_t block_size, num_kv_heads, head_dim, dtype;
  int32_t num_seqs, num_q_heads;
  int32_t n_items, s_max, cf_rows, n_pseudo, pseudo_max_blocks, n_states;
  int64_t decode_ctas;
  uint64_t items_off, cf_ids_off, ptab_off, plen_off, pq_off, seqptr_off, states_off, plan_bytes;
  uint64_t ws_lse_off, ws_dec_off, ws_bytes;
  uint64_t dec_pre_off, dec_lse_off, dec_o_off, dec_total;
};
static_assert(sizeof(TreePlanHeader) <= kTreePlanHeader, "plan header fits its section");

// The chunk-first phase's shapes: bf16 tensor cores, whole or sliced blocks
// per 128-key tile.
bool prefix_tc_shape(const pkv_cache_desc* c, int32_t num_q_heads) {
  if (check_attention_shape(c, num_q_heads) != PKV_OK || c->dtype != PKV_BF16) return false;
  const int P = c->block_size;
  return pkv::kPrefixKeys % P == 0 || P % pkv::kPrefixKeys == 0;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

extern "C" {

pkv_status pkv_chunk_tree_plan(const pkv_cache_desc* cache, const pkv_chunk* chunks,
                               int32_t num_chunks, const int32_t* block_ids,
                               int64_t num_block_ids, int32_t num_seqs, int32_t num_q_heads,
                               int32_t threshold, void* plan, size_t plan_capacity,
                               size_t* plan_bytes, size_t* workspace_bytes) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if ((st = check_attention_shape(cache, num_q_heads)) != PKV_OK) return st;
  if (num_chunks < 0 || num_seqs < 0 || num_block_ids < 0) return PKV_ERR_INVALID_ARG;
  if ((num_chunks > 0 && !chunks) || (num_block_ids > 0 && !block_ids)) return PKV_ERR_INVALID_ARG;
  if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
  const int64_t P = cache->block_size, Hkv = cache->num_kv_heads, Hq = num_q_heads;
  const int G = num_q_heads / cache->num_kv_heads;
  const int RPB = pkv::kPrefixRows / G;  // requests per 128-row query tile
  for (int64_t i = 0; i < num_block_ids; ++i)
    if (block_ids[i] < 0 || block_ids[i] >= cache->num_blocks) return PKV_ERR_INVALID_ARG;
  const bool tc = prefix_tc_shape(cache, num_q_heads);
  const int64_t thr = threshold < 0 ? 1 : threshold;

  // ---- classify the chunks; lay out partial rows, ids and segments
  std::vector<int64_t> where((size_t)num_chunks), ids_at((size_t)num_chunks);
  std::vector<char> first((size_t)num_chunks);
  int64_t cf_rows = 0, cf_ids = 0, n_pseudo = 0, pmax = 0, max_tiles = 0;
  for (int32_t c = 0; c < num_chunks; ++c) {
    const pkv_chunk& k = chunks[c];
    if (k.len < 1 || k.seq_begin < 0 || k.seq_begin >= k.seq_end || k.seq_end > num_seqs ||
        k.first_id < 0 || k.first_id + ceil_div(k.len, P) > num_block_ids)
      return PKV_ERR_INVALID_ARG;
    const int64_t cov = k.seq_end - k.seq_begin, nb = ceil_div(k.len, P);
    first[c] = tc && cov > thr;
    if (first[c]) {
      where[c] = cf_rows;  // a chunk's rows start a query tile: its stores stay inside
      cf_rows += ceil_div(cov, RPB) * RPB;
      ids_at[c] = cf_ids;
      cf_ids += nb;
      max_tiles = std::max(max_tiles, ceil_div(k.len, pkv::kPrefixKeys));
    } else {
      where[c] = n_pseudo;
      n_pseudo += cov;
      pmax = std::max(pmax, nb);
    }
  }
  if (cf_rows > INT32_MAX || cf_ids > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  if (n_pseudo > 65535) return PKV_ERR_UNSUPPORTED;

  // ---- key split of the chunk-first phase: the fewest 128-key tiles per
  // split whose (item x kv head) CTAs still fit one wave on the SMs
  auto count_items = [&](int64_t per) {
    int64_t items = 0;
    for (int32_t c = 0; c < num_chunks; ++c)
      if (first[c])
        items += ceil_div(chunks[c].seq_end - chunks[c].seq_begin, 2 * RPB) *
                 ceil_div(ceil_div(chunks[c].len, pkv::kPrefixKeys), per);
    return items;
  };
  int64_t per = 1, n_items = 0, s_max = 0;
  if (max_tiles > 0) {
    int64_t lo = 1, hi = max_tiles;  // count_items does not grow with per
    const int64_t wave = sm_count();
    while (lo < hi) {
      const int64_t mid = (lo + hi) / 2;
      if (count_items(mid) * Hkv <= wave) hi = mid; else lo = mid + 1;
    }
    per = lo;
    n_items = count_items(per);
    for (int32_t c = 0; c < num_chunks; ++c)
      if (first[c]) s_max = std::max(s_max, ceil_div(chunks[c].len, per * pkv::kPrefixKeys));
  }
  if (n_items > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  const int64_t split_len = per * pkv::kPrefixKeys;
  // states each sequence merges: every key split of a chunk-first chunk on
  // its path, one per other chunk
  int64_t n_states = 0;
  for (int32_t c = 0; c < num_chunks; ++c)
    n_states += (int64_t)(chunks[c].seq_end - chunks[c].seq_begin) *
                (first[c] ? ceil_div(chunks[c].len, split_len) : 1);
  if (n_states > INT32_MAX) return PKV_ERR_UNSUPPORTED;

  // ---- sizes
  TreePlanHeader h{};
  h.magic = kTreePlanMagic;
  h.version = kTreePlanVersion;
  h.num_blocks = cache->num_blocks;
  h.block_size = cache->block_size;
  h.num_kv_heads = cache->num_kv_heads;
  h.head_dim = cache->head_dim;
  h.dtype = cache->dtype;
  h.num_seqs = num_seqs;
  h.num_q_heads = num_q_heads;
  h.n_items = (int32_t)n_items;
  h.s_max = (int32_t)s_max;
  h.cf_rows = (int32_t)cf_rows;
  h.n_pseudo = (int32_t)n_pseudo;
  h.pseudo_max_blocks = (int32_t)pmax;
  h.n_states = (int32_t)n_states;
  h.decode_ctas = n_pseudo > 0 ? decode_ctas(cache, (int32_t)n_pseudo, num_q_heads, (int32_t)pmax, 0)
                               : 0;
  if (h.decode_ctas > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  size_t off = kTreePlanHeader;
  auto section = [&](uint64_t* at, size_t bytes) {
    *at = off;
    off += align256(bytes);
  };
  section(&h.items_off, (size_t)n_items * sizeof(pkv::PrefixItem));
  section(&h.cf_ids_off, (size_t)cf_ids * 4);
  section(&h.ptab_off, (size_t)(n_pseudo * pmax) * 4);
  section(&h.plen_off, (size_t)n_pseudo * 4);
  section(&h.pq_off, (size_t)n_pseudo * 4);
  section(&h.seqptr_off, (size_t)(num_seqs + 1) * 4);
  section(&h.states_off, (size_t)n_states * 16);
  h.plan_bytes = off;
  const int64_t n_ws_states = cf_rows * Hq * s_max + n_pseudo * Hq;  // in the workspace
  h.ws_lse_off = align256((size_t)n_ws_states * cache->head_dim * 4);
  h.ws_dec_off = h.ws_lse_off + align256((size_t)n_ws_states * 4);
  DecodeWorkspace dw{};
  if (n_pseudo > 0) dw = decode_workspace(n_pseudo, h.decode_ctas, G, cache->head_dim);
  h.dec_pre_off = dw.pre_off;
  h.dec_lse_off = dw.lse_off;
  h.dec_o_off = dw.o_off;
  h.dec_total = dw.total;
  h.ws_bytes = h.ws_dec_off + dw.total;
  if (plan_bytes) *plan_bytes = h.plan_bytes;
  if (workspace_bytes) *workspace_bytes = h.ws_bytes;
  if (!plan) return PKV_OK;
  if (plan_capacity < h.plan_bytes) return PKV_ERR_CAPACITY;

  // ---- fill
  unsigned char* base = static_cast<unsigned char*>(plan);
  memset(base, 0, h.plan_bytes);
  memcpy(base, &h, sizeof(h));
  auto* items = reinterpret_cast<pkv::PrefixItem*>(base + h.items_off);
  auto* cfi = reinterpret_cast<int32_t*>(base + h.cf_ids_off);
  auto* ptab = reinterpret_cast<int32_t*>(base + h.ptab_off);
  auto* plen = reinterpret_cast<int32_t*>(base + h.plen_off);
  auto* pq = reinterpret_cast<int32_t*>(base + h.pq_off);
  auto* sptr = reinterpret_cast<int32_t*>(base + h.seqptr_off);
  auto* sref = reinterpret_cast<int64_t*>(base + h.states_off);
  int64_t it = 0;
  for (int32_t c = 0; c < num_chunks; ++c) {
    const pkv_chunk& k = chunks[c];
    const int64_t cov = k.seq_end - k.seq_begin, nb = ceil_div(k.len, P);
    if (first[c]) {
      memcpy(cfi + ids_at[c], block_ids + k.first_id, (size_t)nb * 4);
      for (int64_t r0 = 0; r0 < cov; r0 += 2 * RPB)
        for (int64_t key0 = 0; key0 < k.len; key0 += split_len) {
          pkv::PrefixItem& w = items[it++];
          w.ids_off = (int32_t)ids_at[c];
          w.key0 = (int32_t)key0;
          w.nkeys = (int32_t)std::min<int64_t>(split_len, k.len - key0);
          w.req0 = (int32_t)(k.seq_begin + r0);
          w.nreq = (int32_t)std::min<int64_t>(2 * RPB, cov - r0);
          w.st_req0 = (int32_t)(where[c] + r0);
          w.split = (int32_t)(key0 / split_len);
        }
    } else {
      for (int64_t j = 0; j < cov; ++j) {
        const int64_t p = where[c] + j;
        int32_t* row = ptab + p * pmax;
        memcpy(row, block_ids + k.first_id, (size_t)nb * 4);
        for (int64_t b = nb; b < pmax; ++b) row[b] = -1;
        plen[p] = k.len;
        pq[p] = (int32_t)(k.seq_begin + j);
      }
    }
  }
  // longest work first: the CTAs launch in item order
  std::stable_sort(items, items + n_items, [](const pkv::PrefixItem& x, const pkv::PrefixItem& y) {
    return x.nkeys * (x.nreq + 0LL) > y.nkeys * (y.nreq + 0LL);
  });
  // each sequence's states, in tree order: count, then place
  std::vector<int32_t> fill((size_t)num_seqs + 1, 0);
  for (int32_t c = 0; c < num_chunks; ++c) {
    const int32_t k = first[c] ? (int32_t)ceil_div(chunks[c].len, split_len) : 1;
    for (int32_t r = chunks[c].seq_begin; r < chunks[c].seq_end; ++r) fill[(size_t)r + 1] += k;
  }
  for (int32_t r = 0; r < num_seqs; ++r) fill[(size_t)r + 1] += fill[(size_t)r];
  memcpy(sptr, fill.data(), (size_t)(num_seqs + 1) * 4);
  for (int32_t c = 0; c < num_chunks; ++c) {
    const pkv_chunk& k = chunks[c];
    for (int32_t r = k.seq_begin; r < k.seq_end; ++r) {
      if (first[c]) {  // ((row * Hq + h) * s_max + split)
        const int64_t row = where[c] + (r - k.seq_begin);
        for (int64_t s = 0; s < ceil_div(k.len, split_len); ++s) {
          int64_t* e = sref + 2 * (int64_t)fill[(size_t)r]++;
          e[0] = row * Hq * s_max + s;
          e[1] = s_max;
        }
      } else {  // after every chunk-first state: (segment * Hq + h)
        int64_t* e = sref + 2 * (int64_t)fill[(size_t)r]++;
        e[0] = cf_rows * Hq * s_max + (where[c] + (r - k.seq_begin)) * Hq;
        e[1] = 1;
      }
    }
  }
  return PKV_OK;
}

pkv_status pkv_chunk_tree_attention(const pkv_cache_desc* cache, void* out, float* lse,
                                    const void* q, const void* k_cache, const void* v_cache,
                                    int32_t num_seqs, int32_t num_q_heads, float scale,
                                    const void* plan_host, const void* plan_device,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if ((st = check_attention_shape(cache, num_q_heads)) != PKV_OK) return st;
  if (!plan_host || !plan_device || !isfinite(scale) || num_seqs < 0) return PKV_ERR_INVALID_ARG;
  TreePlanHeader h;
  memcpy(&h, plan_host, sizeof(h));
  if (h.magic != kTreePlanMagic || h.version != kTreePlanVersion ||
      h.num_blocks != cache->num_blocks || h.block_size != cache->block_size ||
      h.num_kv_heads != cache->num_kv_heads || h.head_dim != cache->head_dim ||
      h.dtype != cache->dtype || h.num_seqs != num_seqs || h.num_q_heads != num_q_heads)
    return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(plan_device) & 255u) || workspace_bytes < h.ws_bytes ||
      (h.ws_bytes > 0 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))))
    return PKV_ERR_INVALID_ARG;
  unsigned int* err = device_error_word();
  if (!err) return PKV_ERR_CUDA;
  const int G = num_q_heads / cache->num_kv_heads;
  const float qscale = scale * 1.4426950408889634f;
  const unsigned char* dplan = static_cast<const unsigned char*>(plan_device);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  float* st_o = reinterpret_cast<float*>(ws);
  float* st_lse = reinterpret_cast<float*>(ws + h.ws_lse_off);
  const int64_t cf_states = (int64_t)h.cf_rows * num_q_heads * h.s_max;
  cudaStream_t s = as_stream(stream);

  if (h.n_items > 0) {  // chunk-first: every shared chunk on the tensor cores
    CUtensorMap tmq, ptk, ptv, pto;
    if ((st = encode_q_map_sw128(&tmq, q, num_seqs, num_q_heads, cache->head_dim, G,
                                 pkv::kPrefixRows / G)) != PKV_OK)
      return st;
    if ((st = encode_prefix_maps(&ptk, &ptv, cache, k_cache, v_cache)) != PKV_OK) return st;
    if ((st = encode_prefix_out_map(&pto, st_o, h.cf_rows, cache->num_kv_heads, G, h.s_max,
                                    cache->head_dim)) != PKV_OK)
      return st;
    pkv::PrefixArgs pa{};
    pa.prefix_block_ids = reinterpret_cast<const int32_t*>(dplan + h.cf_ids_off);
    pa.items = reinterpret_cast<const pkv::PrefixItem*>(dplan + h.items_off);
    pa.num_items = h.n_items;
    pa.part_o = st_o;
    pa.part_lse = st_lse;
    pa.err = err;
    pa.num_blocks = cache->num_blocks;
    pa.num_seqs = num_seqs;
    pa.num_q_heads = num_q_heads;
    pa.num_kv_heads = cache->num_kv_heads;
    pa.block_size = cache->block_size;
    pa.parts_stride = h.s_max;
    pa.qscale = qscale;
    pa.lse_scale = 1.f;
    if (pkv::launch_prefix_attention(cache->head_dim, G, 0, tmq, ptk, ptv, pto, pa, s) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
  }
  if (h.n_pseudo > 0) {  // sequence-first: one decode segment per (sequence, chunk)
    pkv::DecodeArgs a{};
    a.q = q;
    a.q_rows = reinterpret_cast<const int32_t*>(dplan + h.pq_off);
    a.block_tables = reinterpret_cast<const int32_t*>(dplan + h.ptab_off);
    a.seq_lens = reinterpret_cast<const int32_t*>(dplan + h.plen_off);
    a.out = nullptr;  // states only
    a.err = err;
    DecodeWorkspace dw{h.dec_pre_off, h.dec_lse_off, h.dec_o_off, h.dec_total};
    bind_decode_workspace(&a, ws + h.ws_dec_off, dw);
    a.st_o = st_o + cf_states * cache->head_dim;
    a.st_lse = st_lse + cf_states;
    a.st_stride = 1;
    a.st_slot = 0;
    a.num_blocks = cache->num_blocks;
    a.max_blocks = h.pseudo_max_blocks;
    a.num_seqs = h.n_pseudo;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = cache->num_kv_heads;
    a.block_size = cache->block_size;
    a.num_ctas = (int32_t)h.decode_ctas;
    a.num_stages = pkv::decode_num_stages(cache->head_dim, elem_bytes(cache->dtype));
    a.qscale = qscale;
    a.plan_before_wait = h.n_items > 0;  // right after the chunk-first prefix kernel
    if ((st = launch_decode(cache, G, q, k_cache, v_cache, a, s, num_seqs)) != PKV_OK) return st;
  }
  pkv::TreeMergeArgs m{};
  m.st_o = st_o;
  m.st_lse = st_lse;
  m.seq_ptr = reinterpret_cast<const int32_t*>(dplan + h.seqptr_off);
  m.states = reinterpret_cast<const int64_t*>(dplan + h.states_off);
  m.out = out;
  m.lse_out = lse;
  m.num_seqs = num_seqs;
  m.num_q_heads = num_q_heads;
  return pkv::launch_tree_merge(cache->dtype, cache->head_dim, m, s) == cudaSuccess ? PKV_OK
                                                                                   : PKV_ERR_CUDA;
}

}  // extern "C"
