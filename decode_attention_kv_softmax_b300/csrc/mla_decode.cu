// MLA absorbed decode (placeholder until the tensor-core kernel lands).
#include "common.cuh"
#include "kernels.h"

extern "C" {
size_t kvdec_mla_workspace_bytes(const kvdec_mla_params*) { return 0; }
kvdec_status kvdec_mla_decode_absorbed(const kvdec_mla_params*, void*) { return KVDEC_ERR_UNSUPPORTED; }
}
