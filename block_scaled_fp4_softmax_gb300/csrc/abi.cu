// Status strings and record geometry of the C ABI.
#include "common.cuh"

extern "C" {

size_t moe_expert_record_bytes(moe_expert_shape s) {
  if (!moe::shape_ok(s)) return 0;
  return moe::record_offsets(s.hidden, s.inter, s.format).total;
}

int moe_expert_record_offsets(moe_expert_shape s, size_t* offsets) {
  if (!offsets) return MOE_ERR_INVALID_ARG;
  if (!moe::shape_ok(s)) return MOE_ERR_UNSUPPORTED;
  moe::RecordOffsets o = moe::record_offsets(s.hidden, s.inter, s.format);
  offsets[0] = o.gate;
  offsets[1] = o.up;
  offsets[2] = o.down;
  offsets[3] = o.gate_s;
  offsets[4] = o.up_s;
  offsets[5] = o.down_s;
  offsets[6] = o.total;
  return MOE_OK;
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or format";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

}  // extern "C"
