// sdm_write_read_noalloc: the forward write/read for callers that cannot allocate device
// memory (see include/sdm.h). Its scratch is one file-scope __device__ array of
// SDM_NOALLOC_SCRATCH_BYTES, which the CUDA driver places when it loads this file's module;
// the call itself allocates nothing and hands the array's device address to the same launch
// sequence sdm_write_read runs, with the slab size chosen so that the workspace fits.
#include "sdm_internal.cuh"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[SDM_NOALLOC_SCRATCH_BYTES];

// The device address of the static scratch on the current device. Host code only holds a
// host-side stand-in for the symbol, so the address is asked from the runtime, with the device
// current, on every call: the lookup is a cheap host call once the array is resident, and a new
// context (after cudaDeviceReset, say) gets its own address instead of a stale one. Under lazy
// module loading the first lookup on a device is what makes the driver load the array.
int scratch_address(void **out) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return (int)e;
    *out = p;
    return 0;
}

}  // namespace

extern "C" int sdm_write_read_noalloc(const sdm_shape *shape, void *bank,
                                      const int32_t *write_slots, const void *write_w,
                                      const float *log_decay, const float *beta, const void *v,
                                      const int32_t *read_slots, const void *read_w,
                                      const int32_t *valid_tokens, void *readings,
                                      void *stream) {
    if (!shape) return sdm_write_read(shape, nullptr, nullptr, nullptr, nullptr, nullptr,
                                      nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 0,
                                      stream);
    sdm_shape s = *shape;
    const size_t cap = SDM_NOALLOC_SCRATCH_BYTES;
    if (s.slab_steps == 0) {
        // the largest slab (in steps) whose workspace fits the static scratch
        const long long nt = s.T >= 1 && s.C >= 1 ? ((long long)s.T + s.C - 1) / s.C : 1;
        int lo = 1, hi = nt > 0 && nt < (1LL << 30) ? (int)nt : 1;
        s.slab_steps = 1;
        const size_t one = sdm_workspace_bytes(&s);
        if (one == 0) return sdm_write_read(&s, bank, write_slots, write_w, log_decay, beta, v,
                                            read_slots, read_w, valid_tokens, readings, nullptr,
                                            0, stream);   // refused shape: its own message
        if (one > cap) {
            return sdm::set_error(SDM_ERR_WORKSPACE,
                                  "sdm_write_read_noalloc: this shape needs %zu bytes of scratch "
                                  "even at one step per slab; the static scratch holds %zu bytes "
                                  "(use sdm_write_read with a caller workspace)", one, cap);
        }
        while (lo < hi) {
            const int mid = lo + (hi - lo + 1) / 2;
            s.slab_steps = mid;
            if (sdm_workspace_bytes(&s) <= cap) lo = mid; else hi = mid - 1;
        }
        s.slab_steps = lo;
    } else {
        const size_t need = sdm_workspace_bytes(&s);
        if (need == 0)   // refused shape: its own message
            return sdm_write_read(&s, bank, write_slots, write_w, log_decay, beta, v, read_slots,
                                  read_w, valid_tokens, readings, nullptr, 0, stream);
        if (need > cap) {
            return sdm::set_error(SDM_ERR_WORKSPACE,
                                  "sdm_write_read_noalloc: slab_steps=%d needs %zu bytes of "
                                  "scratch; the static scratch holds %zu bytes", s.slab_steps,
                                  need, cap);
        }
    }
    void *scratch = nullptr;
    const int e = scratch_address(&scratch);
    if (e)
        return sdm::set_error(SDM_ERR_CUDA, "sdm_write_read_noalloc: static scratch address: %s",
                              cudaGetErrorString((cudaError_t)e));
    return sdm_write_read(&s, bank, write_slots, write_w, log_decay, beta, v, read_slots, read_w,
                          valid_tokens, readings, scratch, cap, stream);
}

extern "C" int sdm_noalloc_get_device_status(sdm_device_status *status, void *stream) {
    if (!status) return sdm::set_error(SDM_ERR_INVALID, "status must not be NULL");
    void *scratch = nullptr;
    const int e = scratch_address(&scratch);
    if (e)
        return sdm::set_error(SDM_ERR_CUDA, "sdm_noalloc_get_device_status: static scratch "
                              "address: %s", cudaGetErrorString((cudaError_t)e));
    // the status block sits at the start of the scratch, as it does in a caller workspace
    return sdm_get_device_status(scratch, status, stream);
}
