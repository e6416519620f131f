// timing.cu -- opt-in launch timing of the attention calls.
//
// Instrumentation for kernel-level rooflines, not part of the attention
// method: while enabled, every decode / prefill / K2/V4 decode call records
// three CUDA events on its stream -- before its partial kernel, before its
// merge, after its merge -- into the next slot of a ring.  Recording between
// the two kernels ends the programmatic overlap of the merge with the partial
// kernel's tail, so a timed run with this on is a separate measurement from an
// untimed one.
//
// Also the testing hook of the kernels' bounded waits (kvq_test_stall_waits):
// a process-wide poll count that the tensor-core attention launches read.
#include <vector>

#include "kvq_internal.cuh"

namespace kvq {
namespace {

struct LaunchTiming {
    std::vector<cudaEvent_t> ev;   // 3 per slot
    std::vector<char> done;        // slot holds all three records
    int32_t cap = 0, next = 0, cur = -1;
};
LaunchTiming g_timing;
int64_t g_stall_polls = 0;

void timing_free() {
    for (cudaEvent_t e : g_timing.ev) cudaEventDestroy(e);
    g_timing.ev.clear();
    g_timing.done.clear();
    g_timing.cap = 0;
    g_timing.next = 0;
    g_timing.cur = -1;
}

}  // namespace

int64_t test_stall_polls() { return g_stall_polls; }
void set_test_stall_polls(int64_t polls) { g_stall_polls = polls; }

void timing_mark(cudaStream_t stream, int phase) {
    LaunchTiming& t = g_timing;
    if (t.cap == 0) return;
    if (phase == 0) {
        t.cur = t.next;
        t.next = (t.next + 1) % t.cap;
        t.done[t.cur] = 0;
    } else if (t.cur < 0) {
        return;   // a merge of a call that was not opened (timing enabled mid-call)
    }
    if (cudaEventRecord(t.ev[3 * t.cur + phase], stream) != cudaSuccess) {
        t.cur = -1;
        return;
    }
    if (phase == 2) {
        t.done[t.cur] = 1;
        t.cur = -1;
    }
}

}  // namespace kvq

extern "C" {

kvq_status kvq_timing_enable(int32_t capacity) {
    using kvq::g_timing;
    if (capacity < 0) return KVQ_ERR_ARG;
    kvq::timing_free();
    if (capacity == 0) return KVQ_OK;
    g_timing.ev.assign(3 * (size_t)capacity, nullptr);
    for (cudaEvent_t& e : g_timing.ev) {
        if (cudaEventCreate(&e) != cudaSuccess) {
            e = nullptr;
            kvq::timing_free();
            return KVQ_ERR_CUDA;
        }
    }
    g_timing.done.assign((size_t)capacity, 0);
    g_timing.cap = capacity;
    return KVQ_OK;
}

kvq_status kvq_timing_read(double* partial_ms, double* merge_ms, int32_t* n_calls) {
    using kvq::g_timing;
    if (!partial_ms || !merge_ms || !n_calls) return KVQ_ERR_ARG;
    *partial_ms = 0.0;
    *merge_ms = 0.0;
    *n_calls = 0;
    for (int32_t s = 0; s < g_timing.cap; ++s) {
        if (!g_timing.done[s]) continue;
        cudaEvent_t* e = &g_timing.ev[3 * (size_t)s];
        float a = 0.0f, b = 0.0f;
        if (cudaEventSynchronize(e[2]) != cudaSuccess || cudaEventElapsedTime(&a, e[0], e[1]) != cudaSuccess ||
            cudaEventElapsedTime(&b, e[1], e[2]) != cudaSuccess)
            return KVQ_ERR_CUDA;
        *partial_ms += a;
        *merge_ms += b;
        ++*n_calls;
        g_timing.done[s] = 0;
    }
    g_timing.next = 0;
    g_timing.cur = -1;
    return KVQ_OK;
}

}  // extern "C"
