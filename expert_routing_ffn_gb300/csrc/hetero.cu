// Heterogeneous CPU-GPU execution of missing experts (SPICE write-up, section
// on CPU-GPU collaboration for prefetch misses, Fig. 6 and its cost model).
//
// A high-confidence miss must be computed exactly.  Per missing expert the
// cost model compares fetching it (its weights over the link, then its FFN on
// the GPU) with running it on the host cores from the host copy of its
// weights (only the token rows cross the link).  This file holds
//   - the device step that applies the decision to the slots of a batch
//     (hetero_decide_kernel) and places the host slots after the GPU
//     segments of the permutation;
//   - the threshold form of the cost model (moe_hetero_fetch_min_rows);
//   - the host side: the exact SwiGLU expert FFN of the host slots on a
//     persistent pool of host threads (moe_cpu_experts).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <condition_variable>
#include <cstring>
#include <mutex>
#include <sched.h>
#include <thread>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "plan.cuh"

namespace moe {

// One block.  (1) FETCH slots per expert and the slots the GPU computes;
// (2) per expert: fewer than fetch_min_rows rows -> host; (3) an ordered pass
// over the slots relabels the host experts' slots CPU and gives the j-th of
// them (slot order) the permuted position n_gpu + j.
__global__ void __launch_bounds__(1024) hetero_decide_kernel(const int32_t* __restrict__ final_idx,
                                                             int32_t* __restrict__ final_kind, int n_slots, int N,
                                                             int fetch_min_rows, uint64_t* __restrict__ fetch_mask,
                                                             uint64_t* __restrict__ cpu_mask,
                                                             int32_t* __restrict__ perm,
                                                             int32_t* __restrict__ inv_perm,
                                                             int32_t* __restrict__ counters) {
    grid_dep_wait();  // the selection's outputs (dependent launch)
    __shared__ int rows[kMaxExperts];
    __shared__ int s_gpu, s_cpu_slots;
    __shared__ unsigned long long s_fetch, s_cpu;
    const int tid = threadIdx.x;
    for (int e = tid; e < kMaxExperts; e += blockDim.x) rows[e] = 0;
    if (tid == 0) { s_gpu = 0; s_cpu_slots = 0; s_fetch = 0ull; s_cpu = 0ull; }
    __syncthreads();
    int gpu = 0;
    for (int i = tid; i < n_slots; i += blockDim.x) {
        const int e = final_idx[i], kd = final_kind[i];
        if (e < 0 || e >= N) continue;
        if (kd == MOE_KIND_FETCH) atomicAdd(&rows[e], 1);
        if (kd == MOE_KIND_COMPUTE || kd == MOE_KIND_FETCH) ++gpu;
    }
    for (int o = 16; o > 0; o >>= 1) gpu += __shfl_xor_sync(0xffffffffu, gpu, o);
    if ((tid & 31) == 0 && gpu) atomicAdd(&s_gpu, gpu);
    __syncthreads();
    if (tid < N && rows[tid] > 0) {
        if (rows[tid] >= fetch_min_rows) {
            atomicOr(&s_fetch, 1ull << tid);
        } else {
            atomicOr(&s_cpu, 1ull << tid);
            atomicAdd(&s_cpu_slots, rows[tid]);
        }
    }
    __syncthreads();
    const unsigned long long host = s_cpu;
    const int n_gpu = s_gpu - s_cpu_slots;
    int base = 0;
    for (int t0 = 0; t0 < n_slots; t0 += blockDim.x) {  // uniform trip count: every thread scans
        const int i = t0 + tid;
        int flag = 0;
        if (i < n_slots) {
            const int e = final_idx[i];
            flag = (e >= 0 && e < N && final_kind[i] == MOE_KIND_FETCH && ((host >> e) & 1ull)) ? 1 : 0;
        }
        int tile = 0;
        const int r = block_exclusive_scan(flag, &tile);
        if (flag) {
            final_kind[i] = MOE_KIND_CPU;
            const int pos = n_gpu + base + r;
            perm[pos] = i;
            inv_perm[i] = pos;
        }
        base += tile;
    }
    if (tid == 0) {
        if (fetch_mask) *fetch_mask = s_fetch;
        if (cpu_mask) *cpu_mask = s_cpu;
        if (counters) {
            counters[MOE_CNT_FETCH] -= s_cpu_slots;
            counters[MOE_CNT_CPU] += s_cpu_slots;
        }
    }
}

cudaError_t launch_hetero_decide(const int32_t* final_idx, int32_t* final_kind, int n_slots, int N,
                                 int fetch_min_rows, uint64_t* fetch_mask, uint64_t* cpu_mask, int32_t* perm,
                                 int32_t* inv_perm, int32_t* counters, cudaStream_t st) {
    return launch_pdl(hetero_decide_kernel, dim3(1), dim3(1024), 0, st, final_idx, final_kind, n_slots, N,
                      fetch_min_rows, fetch_mask, cpu_mask, perm, inv_perm, counters);
}

}  // namespace moe

namespace {

// ---------------------------------------------------------------------------
// Persistent host thread pool.  run(n, threads, fn) calls fn(task) for every
// task in [0, n), spread over at most `threads` threads (the caller is one of
// them), and returns when all tasks are done.  Tasks are taken in index order
// from a shared counter; which thread runs a task does not change its result.
class HostPool {
public:
    static HostPool& get() {
        static HostPool* pool = new HostPool();  // kept until exit: workers never joined
        return *pool;
    }

    int max_threads() const { return (int)workers_.size() + 1; }

    template <typename F>
    void run(int n_tasks, int threads, F& fn) {
        run_erased(n_tasks, threads, &fn, [](void* f, int t) { (*static_cast<F*>(f))(t); });
    }

private:
    void run_erased(int n_tasks, int threads, void* ctx, void (*call)(void*, int)) {
        if (n_tasks <= 0) return;
        std::lock_guard<std::mutex> call_lock(call_mu_);  // one job at a time
        const int helpers = std::max(0, std::min(threads, max_threads()) - 1);
        {
            std::lock_guard<std::mutex> lk(mu_);
            ctx_ = ctx;
            call_ = call;
            n_tasks_ = n_tasks;
            next_.store(0);
            want_ = helpers;
            pending_ = helpers;
            ++generation_;
        }
        cv_work_.notify_all();
        drain();
        std::unique_lock<std::mutex> lk(mu_);
        cv_done_.wait(lk, [&] { return pending_ == 0; });
        ctx_ = nullptr;
    }

    HostPool() {
        int n = 0;
        cpu_set_t set;
        if (sched_getaffinity(0, sizeof(set), &set) == 0) n = CPU_COUNT(&set);
        if (n <= 0) n = (int)std::thread::hardware_concurrency();
        if (n <= 0) n = 1;
        for (int i = 0; i + 1 < n; ++i) workers_.emplace_back([this, i] { loop(i); });
        for (auto& w : workers_) w.detach();
    }

    void drain() {
        for (int t = next_.fetch_add(1); t < n_tasks_; t = next_.fetch_add(1)) call_(ctx_, t);
    }

    void loop(int id) {
        uint64_t seen = 0;
        for (;;) {
            std::unique_lock<std::mutex> lk(mu_);
            cv_work_.wait(lk, [&] { return generation_ != seen; });
            seen = generation_;
            if (id >= want_) continue;
            lk.unlock();
            drain();
            lk.lock();
            if (--pending_ == 0) cv_done_.notify_all();
        }
    }

    std::vector<std::thread> workers_;
    std::mutex call_mu_, mu_;
    std::condition_variable cv_work_, cv_done_;
    void* ctx_ = nullptr;
    void (*call_)(void*, int) = nullptr;
    int n_tasks_ = 0, want_ = 0, pending_ = 0;
    uint64_t generation_ = 0;
    std::atomic<int> next_{0};
};

constexpr int kRowsPerGroup = 8;   // token rows sharing one pass over an expert's weights
constexpr int kMaxHidden = 4096;   // largest d (the ABI's bound for bf16 layers)
constexpr int kChanBlock = 32;     // channels per gate/up task
constexpr int kColBlock = 64;      // output columns per down task

inline float bf16_to_float(uint16_t v) {
    const uint32_t u = (uint32_t)v << 16;
    float f;
    std::memcpy(&f, &u, sizeof(f));
    return f;
}

// One weight row as float32 (bf16 widened exactly).
inline void load_row(const void* base, size_t row, int n, bool bf16, float* out) {
    if (bf16) {
        const uint16_t* p = static_cast<const uint16_t*>(base) + row * (size_t)n;
        for (int j = 0; j < n; ++j) out[j] = bf16_to_float(p[j]);
    } else {
        std::memcpy(out, static_cast<const float*>(base) + row * (size_t)n, sizeof(float) * (size_t)n);
    }
}

// Dot product of two float32 vectors of length n (a multiple of 8): eight
// running sums over j mod 8, added pairwise at the end (a fixed order).
inline float dot8(const float* __restrict__ a, const float* __restrict__ b, int n) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < n; j += 8)
        for (int u = 0; u < 8; ++u) acc[u] += a[j + u] * b[j + u];
    return ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
}

struct Group {  // up to kRowsPerGroup host rows of one expert
    int expert, first, count;  // rows [first, first + count) of the host-row list
};

struct ScratchMap {
    size_t rows, groups, tok_row, x32, h, total;
};

ScratchMap scratch_map(const moe_dims& D) {
    ScratchMap m;
    const size_t slots = (size_t)D.T * D.k;
    size_t o = 0;
    auto take = [&](size_t b) { size_t at = o; o = (o + b + 255) & ~(size_t)255; return at; };
    m.rows = take(slots * 3 * sizeof(int32_t));        // per host row: token, expert, output row
    m.groups = take(slots * sizeof(Group));
    m.tok_row = take((size_t)D.T * sizeof(int32_t));    // token -> its row in x32 (-1: none)
    m.x32 = take((size_t)D.T * D.d * sizeof(float));
    m.h = take(slots * (size_t)D.I * sizeof(float));
    m.total = o;
    return m;
}

bool dims_ok(const moe_dims* D) {
    return D && D->T >= 0 && D->d > 0 && D->d % 8 == 0 && D->d <= kMaxHidden && D->N > 0 && D->N <= 64 &&
           D->k > 0 && D->k <= 8 &&
           D->I > 0 && (D->wtype == MOE_DTYPE_BF16 || D->wtype == MOE_DTYPE_F32);
}

}  // namespace

extern "C" {

int moe_hetero_fetch_min_rows(const moe_hetero_cost* c) {
    if (!c) return -1;
    const double v[5] = {c->link_bytes_per_s, c->expert_bytes, c->gpu_expert_s, c->cpu_row_s, c->hidden_bytes};
    for (double x : v)
        if (!(x >= 0.0) || !std::isfinite(x)) return -1;
    if (!(c->link_bytes_per_s > 0.0)) return -1;
    const double fetch = c->expert_bytes / c->link_bytes_per_s + c->gpu_expert_s;
    // CPU cost of n rows: n t_cpu + 2 n H / B; fetch wins iff fetch < that
    auto cpu = [&](double n) { return n * c->cpu_row_s + 2.0 * (n * c->hidden_bytes) / c->link_bytes_per_s; };
    const double per_row = cpu(1.0);
    if (!(per_row > 0.0)) return INT32_MAX;
    const double q = fetch / per_row;
    if (!(q < 2147483000.0)) return INT32_MAX;
    long n = (long)std::floor(q) + 1;
    // settle rounding at the boundary on the defining inequality itself
    while (n > 1 && fetch < cpu((double)(n - 1))) --n;
    while (!(fetch < cpu((double)n))) ++n;
    return (int)std::max(1L, n);
}

size_t moe_cpu_experts_scratch_size(const moe_dims* dims) {
    if (!dims_ok(dims)) return 0;
    return scratch_map(*dims).total;
}

moe_status moe_cpu_experts(const moe_dims* dims, const void* host_x, const int32_t* host_final_idx,
                           const int32_t* host_final_kind, const void* const* host_w_gate,
                           const void* const* host_w_up, const void* const* host_w_down, int n_threads,
                           float* host_y_rows, void* scratch, size_t scratch_bytes, int32_t* n_rows,
                           int32_t* first_row) {
    if (!dims || !n_rows || !first_row) return MOE_ERR_INVALID_ARG;
    if (!dims_ok(dims)) return MOE_ERR_UNSUPPORTED;
    *n_rows = 0;
    *first_row = 0;
    const moe_dims D = *dims;
    if (D.T == 0) return MOE_OK;
    if (!host_x || !host_final_idx || !host_final_kind || !host_w_gate || !host_w_up || !host_w_down ||
        !host_y_rows || !scratch)
        return MOE_ERR_INVALID_ARG;
    const ScratchMap M = scratch_map(D);
    if (scratch_bytes < M.total) return MOE_ERR_INVALID_ARG;
    const int slots = D.T * D.k, d = D.d, I = D.I;
    const bool bf16 = D.wtype == MOE_DTYPE_BF16;
    char* sb = static_cast<char*>(scratch);
    int32_t* rows = reinterpret_cast<int32_t*>(sb + M.rows);
    Group* groups = reinterpret_cast<Group*>(sb + M.groups);
    int32_t* tok_row = reinterpret_cast<int32_t*>(sb + M.tok_row);
    float* x32 = reinterpret_cast<float*>(sb + M.x32);
    float* h = reinterpret_cast<float*>(sb + M.h);

    // host slots grouped by expert, in slot order within an expert (a
    // counting pass, then placement); GPU slots counted (the y_perm rows
    // before the host rows)
    int per_expert[64] = {0};
    int n_gpu = 0, n = 0;
    for (int s = 0; s < slots; ++s) {
        const int e = host_final_idx[s], kd = host_final_kind[s];
        if (e >= D.N) return MOE_ERR_INVALID_ARG;
        if (e < 0) continue;
        if (kd == MOE_KIND_COMPUTE || kd == MOE_KIND_FETCH) ++n_gpu;
        else if (kd == MOE_KIND_CPU) {
            if (!host_w_gate[e] || !host_w_up[e] || !host_w_down[e]) return MOE_ERR_INVALID_ARG;
            ++per_expert[e];
            ++n;
        }
    }
    *first_row = n_gpu;
    *n_rows = n;
    if (n == 0) return MOE_OK;
    int start[65];
    start[0] = 0;
    for (int e = 0; e < D.N; ++e) start[e + 1] = start[e] + per_expert[e];
    for (int s = 0, j = 0; s < slots; ++s) {
        const int e = host_final_idx[s];
        if (e < 0 || host_final_kind[s] != MOE_KIND_CPU) continue;
        const int at = start[e]++;
        rows[3 * at] = s / D.k;
        rows[3 * at + 1] = e;
        rows[3 * at + 2] = j++;  // output row: rank in slot order
    }
    int n_groups = 0;
    for (int i = 0; i < n;) {
        int j = i;
        while (j < n && rows[3 * j + 1] == rows[3 * i + 1] && j - i < kRowsPerGroup) ++j;
        groups[n_groups++] = Group{rows[3 * i + 1], i, j - i};
        i = j;
    }
    // the tokens' hidden states as float32, once per token
    for (int t = 0; t < D.T; ++t) tok_row[t] = -1;
    int n_tok = 0;
    for (int i = 0; i < n; ++i) {
        const int t = rows[3 * i];
        if (tok_row[t] < 0) {
            tok_row[t] = n_tok;
            load_row(host_x, (size_t)t, d, bf16, x32 + (size_t)n_tok * d);
            ++n_tok;
        }
    }
    const int threads = n_threads > 0 ? n_threads : HostPool::get().max_threads();
    const int cb = (I + kChanBlock - 1) / kChanBlock;
    const int colb = (d + kColBlock - 1) / kColBlock;

    // (1) h[row][c] = SiLU(x . Wg[c]) * (x . Wu[c]), a task per (group, channel block)
    auto gate_up = [&](int task) {
        const Group& g = groups[task / cb];
        const int c0 = (task % cb) * kChanBlock, c1 = std::min(I, c0 + kChanBlock);
        alignas(64) float wg[kMaxHidden], wu[kMaxHidden];
        for (int c = c0; c < c1; ++c) {
            load_row(host_w_gate[g.expert], (size_t)c, d, bf16, wg);
            load_row(host_w_up[g.expert], (size_t)c, d, bf16, wu);
            for (int r = 0; r < g.count; ++r) {
                const int row = g.first + r;
                const float* x = x32 + (size_t)tok_row[rows[3 * row]] * d;
                const float gv = dot8(x, wg, d);
                const float uv = dot8(x, wu, d);
                h[(size_t)row * I + c] = gv / (1.f + std::exp(-gv)) * uv;
            }
        }
    };
    HostPool::get().run(n_groups * cb, threads, gate_up);
    // (2) y[row][j] = sum over channels c, in order, of h[row][c] Wd[c][j],
    //     a task per (group, block of output columns)
    auto down = [&](int task) {
        const Group& g = groups[task / colb];
        const int j0 = (task % colb) * kColBlock, j1 = std::min(d, j0 + kColBlock), w = j1 - j0;
        float acc[kRowsPerGroup][kColBlock];
        for (int r = 0; r < g.count; ++r)
            for (int j = 0; j < w; ++j) acc[r][j] = 0.f;
        float wd[kColBlock];
        for (int c = 0; c < I; ++c) {
            if (bf16) {
                const uint16_t* p = static_cast<const uint16_t*>(host_w_down[g.expert]) + (size_t)c * d + j0;
                for (int j = 0; j < w; ++j) wd[j] = bf16_to_float(p[j]);
            } else {
                const float* p = static_cast<const float*>(host_w_down[g.expert]) + (size_t)c * d + j0;
                for (int j = 0; j < w; ++j) wd[j] = p[j];
            }
            for (int r = 0; r < g.count; ++r) {
                const float hv = h[(size_t)(g.first + r) * I + c];
                for (int j = 0; j < w; ++j) acc[r][j] += hv * wd[j];
            }
        }
        for (int r = 0; r < g.count; ++r) {
            float* y = host_y_rows + (size_t)rows[3 * (g.first + r) + 2] * d + j0;
            for (int j = 0; j < w; ++j) y[j] = acc[r][j];
        }
    };
    HostPool::get().run(n_groups * colb, threads, down);
    return MOE_OK;
}

}  // extern "C"
