// window_idx.cu -- sliding-window ring-slot index rows.
//
// "DeepSeek V4.1", attention/attend, get_window_topk_idxs; "Module attn", window_topk_idxs.
// One thread per output element; each element is a closed form of (query, column), so the
// rows are written straight into their columns of the caller's (possibly wider) index rows.
#include "common.cuh"

namespace dsattn {
namespace {

__global__ void __launch_bounds__(256) window_idx_kernel(int32_t *__restrict__ idx, int64_t ld, int64_t nrows,
                                                         int rows, int cols, int64_t start_pos, int window) {
    // a kernel launched after this one as a programmatic dependent (the attention kernel) may be
    // scheduled as soon as every block of this grid is running; it still waits for this grid to
    // finish (griddepcontrol.wait) before it reads the index rows
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t total = nrows * cols;
    const int oldest = (int)(start_pos % window) + 1;  // decode: slot holding the oldest token
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int j = (int)(e % cols);
        const int64_t r = e / cols;  // bi * rows + q
        int v;
        if (start_pos == 0) {
            // prefill: the causal window of query q, into the chunk itself
            const int q = (int)(r % rows);
            const int first = q - window + 1 > 0 ? q - window + 1 : 0;
            v = first + j;
            if (v > q) v = -1;
        } else {
            // decode: the whole ring, oldest first; a slot past start_pos has not been written yet
            v = oldest + j;
            if (v >= window) v -= window;
            if ((int64_t)v > start_pos) v = -1;
        }
        idx[r * ld + j] = v;
    }
}

}  // namespace

int launch_window_idx(int32_t *idx, int64_t ld, int b, int rows, int cols, int64_t start_pos, int window,
                      cudaStream_t stream) {
    const int64_t nrows = (int64_t)b * rows;
    const int64_t total = nrows * cols;
    if (total == 0) return DS_OK;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    window_idx_kernel<<<(unsigned)blocks, 256, 0, stream>>>(idx, ld, nrows, rows, cols, start_pos, window);
    return launch_status();
}

}  // namespace dsattn
