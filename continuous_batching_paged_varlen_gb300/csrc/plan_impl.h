// The host-side plan object and the planner's entry points.
#pragma once

#include <vector>

#include "../../include/mb.h"
#include "mb_internal.h"

struct mb_plan {
  mb::PlanDevice dev;
  void* workspace = nullptr;
  std::vector<uint8_t> host_image;  // metadata uploaded into the workspace
  int staging = -1;                 // pinned staging buffer of the upload
  mb_plan_info_t info;
};

namespace mb {
mb_status_t validate_config(const mb_config_t* cfg);
mb_status_t validate_requests(const mb_request_t* reqs, int32_t n, const int32_t* bt,
                              const mb_config_t* cfg, int32_t* total_q_out);
mb_status_t build_plan(const mb_request_t* reqs, int32_t n, const int32_t* bt,
                       const mb_config_t* cfg, const mb_plan_options_t* opts,
                       mb_plan* plan);
// page-locked staging buffers for the one host->device copy of a plan
int staging_acquire(int device, size_t bytes);
void* staging_ptr(int idx);
cudaError_t staging_record(int idx, cudaStream_t s);
void staging_release(int idx);
}  // namespace mb
