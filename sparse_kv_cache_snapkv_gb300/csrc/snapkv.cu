// Stage-1 kernels (SnapKV++): placeholder until the tensor-core score kernels land.
#include "rkv_internal.h"

namespace rkv {

void snapkv_plan(int n, int n_kv, int gqa, int max_len, int window, int* nsplit,
                 int* tokens_per_split, int* rows_pad) {
  (void)n; (void)n_kv; (void)gqa; (void)window;
  *nsplit = 1;
  *tokens_per_split = max_len;
  *rows_pad = 128;
}

size_t snapkv_scratch_bytes(int n, int n_kv, int gqa, int max_len, int window) {
  (void)gqa;
  return 2 * align_up((size_t)n * n_kv * (max_len - window) * 4, 256);
}

cudaError_t launch_snapkv(const SnapArgs& a, cudaStream_t s) {
  (void)a; (void)s;
  return cudaErrorNotSupported;
}

}  // namespace rkv
