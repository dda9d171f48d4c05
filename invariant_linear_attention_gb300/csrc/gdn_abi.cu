// gdn_abi.cu -- entry points that are not a kernel launch: workspace sizing,
// the device error word, status strings, and TMA tensor-map encoding.
#include <cudaTypedefs.h>

#include <mutex>

#include "gdn_host.h"

namespace gdn {

size_t fwd_workspace_size(const gdn_shape* s);
size_t bwd_workspace_size(const gdn_shape* s);

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

gdn_status encode_map_3d(CUtensorMap* map, const void* base, gdn_dtype dt, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint32_t b0, uint32_t b2) {
    auto fn = encode_fn();
    if (!fn) return GDN_ERR_CUDA;
    const uint64_t es = elem_size(dt);
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {d0 * es, d0 * d1 * es};
    const cuuint32_t box[3] = {b0, 1u, b2};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = fn(map, dt == GDN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GDN_OK : GDN_ERR_INVALID_ARG;
}

gdn_status encode_rows_sw128(CUtensorMap* map, const void* base, gdn_dtype dt, uint64_t d0, uint64_t d1, uint64_t stride,
                             uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return GDN_ERR_CUDA;
    const cuuint64_t dims[2] = {d0, d1};
    const cuuint64_t strides[1] = {stride};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / elem_size(dt)), box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(map, dt == GDN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GDN_OK : GDN_ERR_INVALID_ARG;
}

}  // namespace gdn

extern "C" size_t gdn_workspace_size(const gdn_shape* shape, int op) {
    using namespace gdn;
    if (check_shape(shape) != GDN_OK) return 0;
    switch (op) {
        case GDN_OP_FWD: return fwd_workspace_size(shape);
        case GDN_OP_DECODE: return 0;
        case GDN_OP_BWD: return bwd_workspace_size(shape);
    }
    return 0;
}

extern "C" gdn_status gdn_read_device_error(void* workspace, unsigned int* bits, void* stream) {
    if (!workspace || !bits) return GDN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned host = 0;
    if (cudaMemcpyAsync(&host, workspace, sizeof(unsigned), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (cudaMemsetAsync(workspace, 0, sizeof(unsigned), s) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
    *bits = host;
    return GDN_OK;
}

extern "C" const char* gdn_status_string(gdn_status status) {
    switch (status) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: null or misaligned pointer, bad shape or aliasing";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: dk/dv/dtype/dv_slice outside the supported set";
        case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA: a CUDA runtime call or kernel launch failed";
    }
    return "unknown gdn_status";
}
