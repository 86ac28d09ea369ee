// ep_launch_model.cu -- host-side SM-count model ("DeepEP Normal vs Low-Latency
// 双模式深度分析", get_theoretical_num_sms of elastic.py), with HBM as the one
// link of a single GPU.
#include <cmath>
#include <cstdint>

#include "../../include/ep.h"

namespace ep {
void record_error(const char* message);
}  // namespace ep

namespace {

double invalid(const char* msg) {
    ep::record_error(msg);
    return -1.0;
}

}  // namespace

// G * (1 - C(E - E/G, k) / C(E, k)); the ratio of binomials is the product over i < k of
// (E - E/G - i) / (E - i), which is 0 once a factor reaches 0.
double ep_expected_topk(int32_t num_groups, int32_t num_experts, int32_t num_topk) {
    if (num_groups < 1 || num_experts < num_groups || num_experts % num_groups != 0)
        return invalid("ep_expected_topk: need 1 <= num_groups <= num_experts and num_experts % num_groups == 0");
    if (num_topk < 1 || num_topk > num_experts) return invalid("ep_expected_topk: need 1 <= num_topk <= num_experts");
    const int64_t outside = num_experts - num_experts / num_groups;  // experts outside one group
    double miss = 1.0;  // probability that no expert of the token falls in a given group
    for (int32_t i = 0; i < num_topk; ++i) {
        const int64_t num = outside - i;
        if (num <= 0) {
            miss = 0.0;
            break;
        }
        miss *= static_cast<double>(num) / static_cast<double>(num_experts - i);
    }
    return num_groups * (1.0 - miss);
}

int32_t ep_theoretical_num_sms(const ep_sm_model* m, int32_t num_ranks, int32_t num_experts, int32_t num_topk,
                               int32_t for_combine) {
    if (m == nullptr) return static_cast<int32_t>(invalid("ep_theoretical_num_sms: model is NULL"));
    if (!(m->hbm_gbs > 0.0) || !(m->sm_read_gbs > 0.0) || !(m->sm_write_gbs > 0.0) || m->num_device_sms < 1)
        return static_cast<int32_t>(
            invalid("ep_theoretical_num_sms: bandwidths must be positive and num_device_sms >= 1"));
    const double rho = ep_expected_topk(num_ranks, num_experts, num_topk);
    if (rho < 0.0) return -1;
    if (rho == 0.0) return m->num_device_sms;  // no traffic
    // per received row: a dispatch reads 1/rho source rows and writes one; a combine the reverse
    const double sm_read = for_combine ? 1.0 : 1.0 / rho;
    const double sm_write = for_combine ? 1.0 / rho : 1.0;
    const double traffic = 1.0 + 1.0 / rho;  // HBM bytes per received row, in rows
    const double rate = m->hbm_gbs / traffic;
    double sms = std::fmax(rate * sm_read / m->sm_read_gbs, rate * sm_write / m->sm_write_gbs);
    int32_t n = static_cast<int32_t>(std::ceil(sms * 1.25));
    n = n < 4 ? 4 : n;
    n = (n + 1) / 2 * 2;
    if (!m->prefer_overlap_with_compute) n = n < 64 ? 64 : n;
    return n < m->num_device_sms ? n : m->num_device_sms;
}
