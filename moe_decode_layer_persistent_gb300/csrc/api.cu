// api.cu -- placeholder C ABI (replaced by the layer implementation).
#include "host_util.h"

extern "C" {
const char* mk_status_string(mk_status s) {
  switch (s) {
    case MK_OK: return "MK_OK";
    case MK_ERR_INVALID_ARG: return "MK_ERR_INVALID_ARG";
    case MK_ERR_UNSUPPORTED: return "MK_ERR_UNSUPPORTED";
    case MK_ERR_CUDA: return "MK_ERR_CUDA";
    case MK_ERR_OOM: return "MK_ERR_OOM";
    case MK_ERR_TIMEOUT: return "MK_ERR_TIMEOUT";
    case MK_ERR_DEVICE_FAULT: return "MK_ERR_DEVICE_FAULT";
  }
  return "MK_ERR_UNKNOWN";
}
mk_status mk_layer_create(const mk_layer_config*, const mk_layer_weights*, mk_layer** out) {
  if (out) *out = nullptr;
  return MK_ERR_UNSUPPORTED;
}
mk_status mk_decode_step(mk_layer*, const mk_step_io*, void*) { return MK_ERR_UNSUPPORTED; }
mk_status mk_layer_status(mk_layer*) { return MK_ERR_UNSUPPORTED; }
mk_status mk_layer_clear_status(mk_layer*) { return MK_ERR_UNSUPPORTED; }
void mk_layer_destroy(mk_layer*) {}
mk_status mk_stack_create(mk_layer* const*, int32_t, mk_stack** out) {
  if (out) *out = nullptr;
  return MK_ERR_UNSUPPORTED;
}
mk_status mk_stack_step(mk_stack*, const mk_stack_io*, void*) { return MK_ERR_UNSUPPORTED; }
mk_status mk_stack_status(mk_stack*) { return MK_ERR_UNSUPPORTED; }
void mk_stack_destroy(mk_stack*) {}
mk_status mk_layer_get_info(mk_layer*, mk_layer_info*) { return MK_ERR_UNSUPPORTED; }
}
