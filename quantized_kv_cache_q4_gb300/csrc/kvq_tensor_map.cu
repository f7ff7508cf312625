// kvq_tensor_map.cu -- TMA descriptors for the code planes of a cache.  The
// driver's encoder is looked up once through the runtime, so the library needs
// no link-time dependency on libcuda.  Encoded descriptors are kept in a small
// table keyed by everything they are made from (plane address, row bytes, row
// count, box height), so a decode step does not pay the driver call again.
#include <cstring>
#include <mutex>

#include "kvq_ptx.cuh"

namespace kvq {
namespace ptx {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static const EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        return EncodeTiledFn(nullptr);
    }();
    return fn;
}

// Codes plane [rows][row_bytes] as a 2D uint8 tensor; box (min(row_bytes, 128)
// bytes, box_rows rows), swizzled over the box width (128, 64 or 32 bytes).
bool encode_codes_map(CUtensorMap *m, void *base, int row_bytes, int64_t rows, int box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int bi = row_bytes < 128 ? row_bytes : 128;
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)bi, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = bi == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : bi == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_32B;
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct MapEntry {
    void *base;
    int row_bytes;
    int box_rows;
    int64_t rows;
    CUtensorMap map;
};

constexpr int kMapSlots = 64;
std::mutex g_map_mutex;
MapEntry g_maps[kMapSlots];
int g_map_used = 0, g_map_next = 0;

}  // namespace

bool make_codes_map(CUtensorMap *m, void *base, int row_bytes, int64_t rows, int box_rows)
{
    {
        std::lock_guard<std::mutex> lock(g_map_mutex);
        for (int i = 0; i < g_map_used; ++i) {
            const MapEntry &e = g_maps[i];
            if (e.base == base && e.row_bytes == row_bytes && e.rows == rows && e.box_rows == box_rows) {
                *m = e.map;
                return true;
            }
        }
    }
    CUtensorMap t;
    std::memset(&t, 0, sizeof t);
    if (!encode_codes_map(&t, base, row_bytes, rows, box_rows)) return false;
    std::lock_guard<std::mutex> lock(g_map_mutex);
    // a full table is overwritten round-robin (an engine keeps a few planes per layer)
    const int slot = g_map_used < kMapSlots ? g_map_used++ : (g_map_next++ % kMapSlots);
    g_maps[slot] = MapEntry{base, row_bytes, box_rows, rows, t};
    *m = t;
    return true;
}

bool tensor_maps_available() { return encode_fn() != nullptr; }

}  // namespace ptx
}  // namespace kvq
