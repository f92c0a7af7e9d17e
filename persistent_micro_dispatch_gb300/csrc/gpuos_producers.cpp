/*
 * Host-thread contention curve of the ring (native producers).
 *
 * "GPUOS: A GPU Operating System Primitive for Transparent Operation Fusion",
 * §3 Q2 "1. Ring Buffer Communication Channel" and §3 Q3 (throughput and
 * scalability) report that ring contention stays small up to about 64
 * concurrent host threads. This program measures that through the C ABI
 * only: T native threads, each committing NOP descriptors in batches of
 * `batch` through one executor's ring, for T = 1, 2, 4, ... up to the given
 * maximum (multi_producer = 1), and the single-producer ring with one thread
 * as the reference. Threads start together at a barrier; the time runs
 * from the barrier to the last thread's last submission, and again to the
 * last completion. One JSON line on stdout.
 *
 * Usage: gpuos_producers [max_threads=64] [per_thread=20000] [batch=16] [device=0]
 */
#include <pthread.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <time.h>

#include <atomic>
#include <vector>

#include "gpuos.h"

namespace {

double now_s()
{
    timespec ts;
    clock_gettime(CLOCK_MONOTONIC, &ts);
    return ts.tv_sec + 1e-9 * ts.tv_nsec;
}

struct Shared {
    gpuos_ctx *ctx = nullptr;
    uint32_t per_thread = 0, batch = 0, threads = 0;
    std::atomic<uint32_t> ready{0};
    std::atomic<uint32_t> go{0};
    std::atomic<int> error{0};
};

void *producer(void *arg)
{
    Shared *sh = static_cast<Shared *>(arg);
    std::vector<gpuos_desc> d(sh->batch);
    memset(d.data(), 0, d.size() * sizeof(gpuos_desc)); /* op 0: NOP */
    sh->ready.fetch_add(1);
    while (!sh->go.load(std::memory_order_acquire)) {
    }
    for (uint32_t i = 0; i < sh->per_thread; i += sh->batch) {
        const int rc = gpuos_submit_batch(sh->ctx, d.data(), sh->batch, nullptr, nullptr, 30000000u);
        if (rc != GPUOS_OK) {
            sh->error.store(rc);
            break;
        }
    }
    return nullptr;
}

/* One row of the curve; returns 0 and fills the rates, or an error code. */
int run(uint32_t T, uint32_t mp, uint32_t per_thread, uint32_t batch, int device, double *submit_rate,
        double *complete_rate)
{
    gpuos_config cfg;
    gpuos_default_config(&cfg);
    cfg.multi_producer = mp;
    cfg.device = device;
    gpuos_ctx *ctx = nullptr;
    int rc = gpuos_init(&cfg, &ctx);
    if (rc) return rc;
    Shared sh;
    sh.ctx = ctx;
    sh.per_thread = per_thread;
    sh.batch = batch;
    sh.threads = T;
    std::vector<pthread_t> th(T);
    for (uint32_t i = 0; i < T; i++) pthread_create(&th[i], nullptr, producer, &sh);
    while (sh.ready.load() < T) {
    }
    const double t0 = now_s();
    sh.go.store(1, std::memory_order_release);
    for (uint32_t i = 0; i < T; i++) pthread_join(th[i], nullptr);
    const double t1 = now_s();
    rc = sh.error.load();
    if (rc == GPUOS_OK) rc = gpuos_sync(ctx, UINT64_MAX, 60000);
    const double t2 = now_s();
    const int sd = gpuos_shutdown(ctx, 30000);
    if (rc == GPUOS_OK) rc = sd;
    const double n = (double)T * (double)(per_thread / batch * batch);
    *submit_rate = n / (t1 - t0);
    *complete_rate = n / (t2 - t0);
    return rc;
}

}  // namespace

int main(int argc, char **argv)
{
    const uint32_t max_t = argc > 1 ? (uint32_t)atoi(argv[1]) : 64u;
    const uint32_t per_thread = argc > 2 ? (uint32_t)atoi(argv[2]) : 20000u;
    const uint32_t batch = argc > 3 ? (uint32_t)atoi(argv[3]) : 16u;
    const int device = argc > 4 ? atoi(argv[4]) : 0;
    if (batch == 0 || batch > 4096 || per_thread < batch || max_t == 0) {
        fprintf(stderr, "usage: gpuos_producers [max_threads] [per_thread] [batch<=4096] [device]\n");
        return 2;
    }
    printf("{\"metric\": \"host submission throughput vs producer threads (native threads, NOP batches of %u)\", "
           "\"unit\": \"descriptors/s\", \"rows\": [",
           batch);
    bool first = true;
    std::vector<std::pair<uint32_t, uint32_t>> plan = {{1u, 0u}};
    for (uint32_t T = 1; T <= max_t; T *= 2) plan.push_back({T, 1u});
    for (auto &pt : plan) {
        double s = 0, c = 0;
        const int rc = run(pt.first, pt.second, per_thread, batch, device, &s, &c);
        if (rc) {
            fprintf(stderr, "gpuos_producers: T=%u mp=%u failed: %s (%d)\n", pt.first, pt.second,
                    gpuos_strerror(rc, 0), rc);
            printf("]}\n");
            return 1;
        }
        printf("%s{\"threads\": %u, \"multi_producer\": %u, \"descriptors\": %u, \"submit_per_s\": %.1f, "
               "\"complete_per_s\": %.1f}",
               first ? "" : ", ", pt.first, pt.second, pt.first * (per_thread / batch * batch), s, c);
        first = false;
        fflush(stdout);
    }
    printf("]}\n");
    return 0;
}
