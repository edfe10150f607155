// Prefill (nt >= 1) for the concat class: tcgen05 bf16 GEMM + per-token epilogue.
#include "qkv_internal.h"

qkv_status launch_prefill(const PrefillParams&, cudaStream_t, const char** why) {
    *why = "the tcgen05 prefill kernel is not built into this library yet";
    return QKV_ERR_UNSUPPORTED;
}
