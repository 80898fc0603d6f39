// Scope guard that times one kernel launch when timing is enabled
// (kda_timing_enable); see kda_timing.cu.
#pragma once

#include <cuda_runtime.h>

namespace kda {

class TimedLaunch {
  public:
    TimedLaunch(const char* name, cudaStream_t s);
    ~TimedLaunch();
    TimedLaunch(const TimedLaunch&) = delete;
    TimedLaunch& operator=(const TimedLaunch&) = delete;

  private:
    const char* name_;
    cudaStream_t s_;
    cudaEvent_t start_ = nullptr, stop_ = nullptr;
    bool active_ = false;
};

}  // namespace kda
