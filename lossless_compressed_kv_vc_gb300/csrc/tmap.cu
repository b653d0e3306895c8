// Host side of the TMA loads: the driver's tensor-map encoder, fetched through the runtime (the
// library does not link the driver API), and a small cache of the row maps the draft step uses.
//
// A draft launch needs two maps per token-drop request (kept K rows, kept V rows). The buffers
// they describe live for many steps, so the maps are built once per (base, rows, d) and reused;
// the cache is cleared when it grows past a bound so that a caller cycling through many buffers
// does not grow it without limit.
#include "vc_internal.cuh"

#include <cudaTypedefs.h>

#include <mutex>
#include <unordered_map>

namespace vc {

void* tmap_encoder() {
  static void* fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = f;
  });
  return fn;
}

namespace {

struct RowsKey {
  uintptr_t base;
  int64_t rows;
  int d;
  bool operator==(const RowsKey& o) const { return base == o.base && rows == o.rows && d == o.d; }
};
struct RowsKeyHash {
  size_t operator()(const RowsKey& k) const {
    size_t h = std::hash<uintptr_t>()(k.base);
    h ^= std::hash<int64_t>()(k.rows) + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
    h ^= std::hash<int>()(k.d) + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
    return h;
  }
};

constexpr size_t kMaxCached = 4096;
std::mutex g_mu;
std::unordered_map<RowsKey, CUtensorMap, RowsKeyHash> g_rows;

}  // namespace

bool rows_tmap(CUtensorMap* out, const void* base, int d, int64_t rows) {
  if (!base || rows < 1 || rows >= (int64_t(1) << 31) || (d != 64 && d != 128)) return false;
  const RowsKey key{reinterpret_cast<uintptr_t>(base), rows, d};
  {
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_rows.find(key);
    if (it != g_rows.end()) {
      *out = it->second;
      return true;
    }
  }
  auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tmap_encoder());
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64, 1};
  cuuint32_t es[2] = {1, 1};
  CUtensorMap m;
  if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_rows.size() >= kMaxCached) g_rows.clear();
  g_rows.emplace(key, m);
  *out = m;
  return true;
}

}  // namespace vc
