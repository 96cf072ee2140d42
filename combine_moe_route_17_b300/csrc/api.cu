// Host-side entry points of the C ABI that launch no kernel of their own:
// shape validation, workspace sizing and set-up, the expert offsets the count
// pass left in the workspace, the device error word and the status strings.
#include "moe_common.cuh"

extern "C" moe_status moe_validate_shape(const moe_shape* shape) { return moe::validate(shape); }

extern "C" moe_status moe_workspace_size(const moe_shape* shape, size_t* bytes) {
    moe_status st = moe::validate(shape);
    if (st != MOE_OK) return st;
    if (!bytes) return MOE_ERR_INVALID_ARG;
    *bytes = moe::ws_layout(*shape).total;
    return MOE_OK;
}

extern "C" moe_status moe_workspace_init(void* workspace, size_t ws_bytes, cudaStream_t stream) {
    if (!workspace || !moe::aligned(workspace, 256) || ws_bytes < sizeof(moe::WsHeader))
        return MOE_ERR_INVALID_ARG;
    return cudaMemsetAsync(workspace, 0, ws_bytes, stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" moe_status moe_expert_offsets(const moe_shape* shape, const void* workspace,
                                         size_t ws_bytes, int32_t* expert_off,
                                         cudaStream_t stream) {
    moe_status st = moe::validate(shape);
    if (st != MOE_OK) return st;
    const moe::WsLayout L = moe::ws_layout(*shape);
    if (!workspace || !moe::aligned(workspace, 256) || ws_bytes < L.total) return MOE_ERR_INVALID_ARG;
    if (!expert_off || !moe::aligned(expert_off, 4)) return MOE_ERR_INVALID_ARG;
    // the table the count pass's finishing CTA scanned from the expert totals
    const size_t n = sizeof(int32_t) * ((size_t)shape->E + 1);
    return cudaMemcpyAsync(expert_off, moe::ws_ptr<int32_t>(workspace, L.eoff), n,
                           cudaMemcpyDeviceToDevice, stream) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

extern "C" moe_status moe_get_device_error(void* workspace, cudaStream_t stream) {
    if (!workspace || !moe::aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
    uint32_t word[2] = {0, 0};
    auto* hdr = moe::ws_ptr<moe::WsHeader>(workspace, 0);
    if (cudaMemcpyAsync(word, &hdr->error, sizeof(word), cudaMemcpyDeviceToHost, stream) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (word[0] != 0) {
        if (cudaMemsetAsync(&hdr->error, 0, sizeof(word), stream) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
    }
    switch (word[0]) {
        case 0: return MOE_OK;
        case MOE_ERR_TIMEOUT: return MOE_ERR_TIMEOUT;
        default: return MOE_ERR_DEVICE_CHECK;
    }
}

extern "C" moe_status moe_debug_set_fault(void* workspace, int tile, uint64_t wait_ns,
                                          cudaStream_t stream) {
    if (!workspace || !moe::aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
    auto* hdr = moe::ws_ptr<moe::WsHeader>(workspace, 0);
    const int32_t p1 = tile < 0 ? 0 : tile + 1;
    if (cudaMemcpyAsync(&hdr->fault_tile_p1, &p1, sizeof(p1), cudaMemcpyHostToDevice, stream) !=
            cudaSuccess ||
        cudaMemcpyAsync(&hdr->wait_ns, &wait_ns, sizeof(wait_ns), cudaMemcpyHostToDevice, stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

extern "C" const char* moe_status_string(moe_status status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_TIMEOUT: return "device wait timed out";
        case MOE_ERR_DEVICE_CHECK: return "device-side check failed";
    }
    return "unknown status";
}

extern "C" int moe_abi_version(void) { return MOE_ROUTE_ABI_VERSION; }
