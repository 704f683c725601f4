// Internal to libssmverify: state shared between its translation units.
#ifndef SSM_INTERNAL_H
#define SSM_INTERNAL_H

namespace ssm_internal {

// Record the CUDA error of the calling thread's last failed launch (what
// ssm_last_cuda_error() returns).
__attribute__((visibility("hidden"))) void set_last_cuda_error(int e);

}  // namespace ssm_internal

#endif  // SSM_INTERNAL_H
