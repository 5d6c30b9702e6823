// eplb.cpp -- expert placement planner (host).
//
// "ep-deploy" handbook page, section "EPLB 与路由约束": experts are placed on
// GPUs in three greedy steps.  Hierarchical: (1) the expert groups are
// packed onto the nodes by group load, the same number of groups per node,
// so a group never spans nodes; (2) inside each node the hottest experts get
// extra physical copies, one at a time to the expert with the largest load
// per copy; (3) the node's physical experts (weight: load / copies) are
// packed onto its GPUs, the same number per GPU.  Global: the cluster is one
// node.  Packing takes items heaviest first (equal weights: lower index
// first) and puts each into the lightest pack that is not full (equal
// loads: lower pack index).
//
// Here the steps run on ordered sets and heaps, O(n log n) per step.
#include <algorithm>
#include <cmath>
#include <numeric>
#include <queue>
#include <set>
#include <utility>
#include <vector>

#include "../../include/moe.h"

namespace {

// packs[p * per + q] = q-th item placed in pack p
void balanced_pack(const std::vector<double> &w, int n_packs, std::vector<int> &packs) {
  const int n = static_cast<int>(w.size());
  const int per = n / n_packs;
  std::vector<int> order(n);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return w[a] > w[b]; });
  std::set<std::pair<double, int>> open;  // (load, pack) of packs with room
  for (int p = 0; p < n_packs; ++p) open.insert({0.0, p});
  std::vector<int> fill(n_packs, 0);
  packs.assign(n, -1);
  for (int it : order) {
    auto best = *open.begin();
    open.erase(open.begin());
    const int p = best.second;
    packs[p * per + fill[p]] = it;
    if (++fill[p] < per) open.insert({best.first + w[it], p});
  }
}

}  // namespace

extern "C" moe_status_t moe_eplb_plan(const double *load, int32_t num_experts,
                                      int32_t num_groups, int32_t num_nodes, int32_t num_gpus,
                                      int32_t num_physical, int32_t *gpu_slots,
                                      int32_t *replicas) {
  const int E = num_experts, groups = num_groups, gpus = num_gpus, phys = num_physical;
  const int n_nodes = num_nodes > 0 ? num_nodes : 1;
  if (!load || !gpu_slots || !replicas) return MOE_ERR_INVALID_ARG;
  if (E <= 0 || groups <= 0 || gpus <= 0 || num_nodes < 0 || E % groups != 0 ||
      groups % n_nodes != 0 || gpus % n_nodes != 0 || phys % gpus != 0 || phys < E)
    return MOE_ERR_INVALID_ARG;
  for (int e = 0; e < E; ++e)
    if (!(load[e] >= 0.0) || !std::isfinite(load[e])) return MOE_ERR_INVALID_ARG;
  const int gsize = E / groups, per_node_e = E / n_nodes;
  const int node_phys = phys / n_nodes, node_gpus = gpus / n_nodes;
  if (node_gpus * (phys / gpus) != node_phys) return MOE_ERR_INVALID_ARG;

  // experts of each node, in the order their groups were packed
  std::vector<int> node_experts(E);
  if (num_nodes > 0) {
    std::vector<double> gload(groups, 0.0);
    for (int g = 0; g < groups; ++g)
      for (int i = 0; i < gsize; ++i) gload[g] += load[g * gsize + i];
    std::vector<int> gpack;
    balanced_pack(gload, num_nodes, gpack);
    const int per_node_g = groups / num_nodes;
    for (int nd = 0; nd < num_nodes; ++nd)
      for (int q = 0; q < per_node_g; ++q) {
        const int g = gpack[nd * per_node_g + q];
        for (int i = 0; i < gsize; ++i)
          node_experts[nd * per_node_e + q * gsize + i] = g * gsize + i;
      }
  } else {
    std::iota(node_experts.begin(), node_experts.end(), 0);
  }

  std::vector<int> cnt(E, 0);
  for (int nd = 0; nd < n_nodes; ++nd) {
    const int *ids = node_experts.data() + nd * per_node_e;
    // replicas: max-heap on (load per copy, then earlier position)
    auto less = [&](int a, int b) {
      const double la = load[ids[a]] / cnt[ids[a]], lb = load[ids[b]] / cnt[ids[b]];
      return la < lb || (la == lb && a > b);
    };
    std::priority_queue<int, std::vector<int>, decltype(less)> heap(less);
    for (int i = 0; i < per_node_e; ++i) {
      cnt[ids[i]] = 1;
      heap.push(i);
    }
    for (int r = per_node_e; r < node_phys; ++r) {
      const int i = heap.top();
      heap.pop();
      cnt[ids[i]] += 1;
      heap.push(i);
    }
    std::vector<int> phys_e;
    std::vector<double> w;
    phys_e.reserve(node_phys);
    w.reserve(node_phys);
    for (int i = 0; i < per_node_e; ++i)
      for (int c = 0; c < cnt[ids[i]]; ++c) {
        phys_e.push_back(ids[i]);
        w.push_back(load[ids[i]] / cnt[ids[i]]);
      }
    std::vector<int> packs;
    balanced_pack(w, node_gpus, packs);
    for (int q = 0; q < node_phys; ++q) gpu_slots[nd * node_phys + q] = phys_e[packs[q]];
  }
  for (int e = 0; e < E; ++e) replicas[e] = cnt[e];
  return MOE_OK;
}
