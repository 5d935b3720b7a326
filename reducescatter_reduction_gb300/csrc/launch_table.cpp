// The launch table CCL_VARIANT_AUTO consults, and its lookup.
//
// T-CCL, section "Launch Configuration Tuning": launch configurations are
// profiled offline and ranked per message size in a table the runtime reads.
// launch_table.inc (written by calibrate.py on the GPU) holds the measured
// per-call device time of the ld/st and the TMA AllReduce at points (p,
// element bytes, SM budget, bytes per rank).  Both kernels give identical
// bits, so the choice changes only the time.
//
// Lookup for a call (p, s, budget, bytes):
//  - the measured rank count nearest to p on a log scale (ties: the larger);
//  - the element size s itself (2 or 4 bytes);
//  - the measured SM budget nearest on a log scale, "every SM" counting as
//    the table's SM count, so a budget at or above the device's SM count is
//    "every SM";
//  - between two measured sizes, a power law through the two times (a
//    straight line on log-log axes); below the smallest, its time (the
//    latency floor); above the largest, the straight line through the last
//    two points (the bandwidth-bound regime).
// AUTO takes TMA when its estimate is below kTmaMargin times the ld/st one.
#include <cmath>
#include <cstddef>
#include <cstdint>

#include "internal.h"

namespace ccl {

namespace {

struct LaunchPoint {
    int p;
    int elem_bytes;
    int sm_budget;            // 0 = every SM
    unsigned long long bytes; // per rank
    float us_ldst;
    float us_tma;
};

#include "launch_table.inc"

constexpr double kTmaMargin = 0.98;

double log_dist(double a, double b) { return std::fabs(std::log2(a) - std::log2(b)); }

// Distinct values of a column among rows matching a filter, nearest to x.
template <typename Key, typename Match>
int nearest(Key key, Match match, double x, int sms)
{
    int best = -1;
    double bd = 1e300;
    for (const LaunchPoint *r = kLaunchTable; r->p != 0; ++r) {
        if (!match(*r)) continue;
        const int v = key(*r);
        const double dv = v == 0 ? double(sms) : double(v);
        const double d = log_dist(dv, x);
        if (d < bd - 1e-12 || (std::fabs(d - bd) <= 1e-12 && v > best)) {
            bd = d;
            best = v;
        }
    }
    return best;
}

double pick(const LaunchPoint &r, int variant) { return variant == CCL_VARIANT_TMA ? r.us_tma : r.us_ldst; }

}  // namespace

bool launch_table_estimate(int p, int elem_bytes, int sm_budget, int num_sms, double bytes_per_rank, int variant,
                           double *us)
{
    if (p < 1 || (elem_bytes != 2 && elem_bytes != 4) || bytes_per_rank < 0 ||
        (variant != CCL_VARIANT_LDST && variant != CCL_VARIANT_TMA))
        return false;
    const int sms = num_sms > 0 ? num_sms : kLaunchTableSms;
    const int budget = (sm_budget <= 0 || sm_budget >= sms) ? 0 : sm_budget;
    const int tp = nearest([](const LaunchPoint &r) { return r.p; },
                           [&](const LaunchPoint &r) { return r.elem_bytes == elem_bytes; }, double(p), sms);
    if (tp < 0) return false;
    const double want_b = budget == 0 ? double(kLaunchTableSms) : double(budget) * kLaunchTableSms / sms;
    const int tb = nearest([](const LaunchPoint &r) { return r.sm_budget; },
                           [&](const LaunchPoint &r) { return r.p == tp && r.elem_bytes == elem_bytes; }, want_b,
                           kLaunchTableSms);
    if (tb < 0) return false;
    // rows of the chosen (p, s, budget), in increasing size (the table is sorted)
    const LaunchPoint *lo = nullptr, *hi = nullptr, *prev = nullptr, *last = nullptr;
    for (const LaunchPoint *r = kLaunchTable; r->p != 0; ++r) {
        if (r->p != tp || r->elem_bytes != elem_bytes || r->sm_budget != tb) continue;
        if (double(r->bytes) <= bytes_per_rank) lo = r;
        if (!hi && double(r->bytes) >= bytes_per_rank) hi = r;
        prev = last;
        last = r;
    }
    if (!last) return false;
    double t;
    if (!lo) {
        t = pick(*hi, variant);                       // below the smallest point: its time
    } else if (!hi) {
        if (!prev) {
            t = pick(*last, variant) * bytes_per_rank / double(last->bytes);
        } else {                                      // above the largest: the line through the last two
            const double slope = (pick(*last, variant) - pick(*prev, variant)) / double(last->bytes - prev->bytes);
            t = pick(*last, variant) + slope * (bytes_per_rank - double(last->bytes));
        }
    } else if (lo == hi || lo->bytes == hi->bytes) {
        t = pick(*lo, variant);
    } else {                                          // power law between the two neighbours
        const double f = std::log(bytes_per_rank / double(lo->bytes)) / std::log(double(hi->bytes) / double(lo->bytes));
        t = std::exp(std::log(pick(*lo, variant)) + f * (std::log(pick(*hi, variant)) - std::log(pick(*lo, variant))));
    }
    *us = t;
    return true;
}

bool launch_table_prefers_tma(int p, int elem_bytes, int sm_budget, int num_sms, double bytes_per_rank)
{
    double ldst = 0, tma = 0;
    if (!launch_table_estimate(p, elem_bytes, sm_budget, num_sms, bytes_per_rank, CCL_VARIANT_LDST, &ldst)) return false;
    if (!launch_table_estimate(p, elem_bytes, sm_budget, num_sms, bytes_per_rank, CCL_VARIANT_TMA, &tma)) return false;
    return tma < kTmaMargin * ldst;
}

int launch_table_points() { int k = 0; for (const LaunchPoint *r = kLaunchTable; r->p != 0; ++r) ++k; return k; }

}  // namespace ccl

extern "C" ccl_status_t ccl_launch_estimate(int p, ccl_dtype_t dtype, int sm_budget, size_t bytes_per_rank, int variant,
                                            double *us)
{
    if (!us) return ccl::record_error(CCL_ERR_INVALID_ARG, "ccl_launch_estimate: us is NULL");
    if (p < 1 || p > ccl::kMaxRanks || dtype < CCL_F32 || dtype > CCL_I32 || sm_budget < 0 ||
        (variant != CCL_VARIANT_LDST && variant != CCL_VARIANT_TMA))
        return ccl::record_error(CCL_ERR_INVALID_ARG, "ccl_launch_estimate: argument out of range");
    if (!ccl::launch_table_estimate(p, int(ccl::elem_bytes(dtype)), sm_budget, 0, double(bytes_per_rank), variant, us))
        return ccl::record_error(CCL_ERR_UNSUPPORTED, "ccl_launch_estimate: the launch table has no point for this");
    return CCL_OK;
}
