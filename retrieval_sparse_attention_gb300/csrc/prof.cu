// prof.cu -- optional CUDA-event bracketing of every kernel launch
// (include/gca_prof.h).
#include <string.h>

#include <string>
#include <vector>

#include "gca_prof.h"
#include "kernels.h"

namespace gca {
namespace {

struct Rec {
    const char* name;
    cudaEvent_t a, b;
};

thread_local bool t_on = false;
thread_local std::vector<Rec> t_recs;
thread_local std::vector<cudaEvent_t> t_pool;
thread_local cudaEvent_t t_open = nullptr;
thread_local const char* t_open_name = nullptr;

cudaEvent_t take_event() {
    if (!t_pool.empty()) {
        cudaEvent_t e = t_pool.back();
        t_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

}  // namespace

void prof_begin(cudaStream_t st, const char* name) {
    if (!t_on) return;
    t_open = take_event();
    t_open_name = name;
    if (t_open) cudaEventRecord(t_open, st);
}

void prof_end(cudaStream_t st) {
    if (!t_on || !t_open) return;
    cudaEvent_t b = take_event();
    if (!b) return;
    cudaEventRecord(b, st);
    t_recs.push_back(Rec{t_open_name, t_open, b});
    t_open = nullptr;
}

}  // namespace gca

using namespace gca;

extern "C" {

void gca_prof_enable(int on) { t_on = on != 0; }

int gca_prof_read(int max, char* names, float* total_ms, int* launches) {
    std::vector<std::string> keys;
    std::vector<float> ms;
    std::vector<int> cnt;
    int rc = 0;
    for (const Rec& r : t_recs) {
        float t = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
            rc = -1;
        size_t i = 0;
        while (i < keys.size() && keys[i] != r.name) ++i;
        if (i == keys.size()) { keys.push_back(r.name); ms.push_back(0.f); cnt.push_back(0); }
        ms[i] += t;
        cnt[i] += 1;
        t_pool.push_back(r.a);
        t_pool.push_back(r.b);
    }
    t_recs.clear();
    if (rc != 0) return -1;
    int n = 0;
    for (size_t i = 0; i < keys.size() && n < max; ++i, ++n) {
        strncpy(names + 64 * n, keys[i].c_str(), 63);
        names[64 * n + 63] = 0;
        total_ms[n] = ms[i];
        launches[n] = cnt[i];
    }
    return n;
}

}  // extern "C"
