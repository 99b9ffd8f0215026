// Owner planning ("MatrixFSDP", section 4.1, Algorithm 1): every role (a 2D
// matrix, or the packed non-matrix tail of a block) is assigned whole to one
// data-parallel rank, balancing owner-resident element counts. Integer work
// only, host only.
#include <algorithm>
#include <cstdint>
#include <numeric>
#include <vector>

#include "mo.h"

namespace {

// Index of the lightest rank (lowest index on ties).
int32_t lightest(const std::vector<int64_t>& load) {
  int32_t best = 0;
  for (int32_t r = 1; r < int32_t(load.size()); ++r)
    if (load[size_t(r)] < load[size_t(best)]) best = r;
  return best;
}

// Roles in decreasing numel, ties kept in table order.
std::vector<int32_t> by_size(const mo_role* roles, const std::vector<int32_t>& subset) {
  std::vector<int32_t> order = subset;
  std::stable_sort(order.begin(), order.end(),
                   [&](int32_t a, int32_t b) { return roles[a].numel > roles[b].numel; });
  return order;
}

void role_greedy(const mo_role* roles, int32_t n, int32_t world, std::vector<int32_t>& owner,
                 std::vector<int64_t>& load) {
  owner.assign(size_t(n), -1);
  load.assign(size_t(world), 0);
  std::vector<int32_t> blocks;
  for (int32_t i = 0; i < n; ++i) blocks.push_back(roles[i].block);
  std::sort(blocks.begin(), blocks.end());
  blocks.erase(std::unique(blocks.begin(), blocks.end()), blocks.end());
  for (int32_t b : blocks) {
    std::vector<int32_t> members;
    for (int32_t i = 0; i < n; ++i)
      if (roles[i].block == b) members.push_back(i);
    for (int32_t i : by_size(roles, members)) {
      const int32_t r = lightest(load);
      owner[size_t(i)] = r;
      load[size_t(r)] += roles[i].numel;
    }
  }
}

void scope_greedy(const mo_role* roles, int32_t n, int32_t world, std::vector<int32_t>& owner,
                  std::vector<int64_t>& load) {
  owner.assign(size_t(n), -1);
  load.assign(size_t(world), 0);
  std::vector<int32_t> all(static_cast<size_t>(n), 0);
  std::iota(all.begin(), all.end(), 0);
  for (int32_t i : by_size(roles, all)) {
    const int32_t r = lightest(load);
    owner[size_t(i)] = r;
    load[size_t(r)] += roles[i].numel;
  }
}

// max/avg of the loads, as a rational compared by cross-multiplication:
// returns true if imbalance(a) < imbalance(b) for equal totals and world.
bool less_imbalanced(const std::vector<int64_t>& a, const std::vector<int64_t>& b) {
  const int64_t ma = *std::max_element(a.begin(), a.end());
  const int64_t mb = *std::max_element(b.begin(), b.end());
  return ma < mb;   // the totals (hence the averages) are equal
}

int64_t max_block_load(const mo_role* roles, int32_t n, int32_t world, const std::vector<int32_t>& owner) {
  std::vector<int32_t> blocks;
  for (int32_t i = 0; i < n; ++i) blocks.push_back(roles[i].block);
  std::sort(blocks.begin(), blocks.end());
  blocks.erase(std::unique(blocks.begin(), blocks.end()), blocks.end());
  int64_t worst = 0;
  for (int32_t b : blocks) {
    std::vector<int64_t> per(size_t(world), 0);
    for (int32_t i = 0; i < n; ++i)
      if (roles[i].block == b) per[size_t(owner[size_t(i)])] += roles[i].numel;
    worst = std::max(worst, *std::max_element(per.begin(), per.end()));
  }
  return worst;
}

}  // namespace

extern "C" int mo_plan_owners(const mo_role* roles, int32_t nroles, int32_t world, int32_t strategy,
                              int64_t block_cap, int32_t* owner_out, int64_t* load_out, int32_t* chosen_out) {
  if (world < 1 || strategy < MO_PLAN_ROLE_GREEDY || strategy > MO_PLAN_COST_AWARE) return MO_ERR_BAD_PARAM;
  if (nroles < 0) return MO_ERR_BAD_SHAPE;
  if (nroles > 0 && (!roles || !owner_out)) return MO_ERR_NULL_POINTER;
  for (int32_t i = 0; i < nroles; ++i)
    if (roles[i].numel < 0 || roles[i].block < 0) return MO_ERR_BAD_SHAPE;
  std::vector<int32_t> owner;
  std::vector<int64_t> load;
  int32_t chosen = strategy;
  if (strategy == MO_PLAN_ROLE_GREEDY) {
    role_greedy(roles, nroles, world, owner, load);
  } else if (strategy == MO_PLAN_SCOPE_GREEDY) {
    scope_greedy(roles, nroles, world, owner, load);
  } else {
    std::vector<int32_t> o_role, o_scope;
    std::vector<int64_t> l_role, l_scope;
    role_greedy(roles, nroles, world, o_role, l_role);
    scope_greedy(roles, nroles, world, o_scope, l_scope);
    const bool within_cap = block_cap <= 0 || max_block_load(roles, nroles, world, o_scope) <= block_cap;
    if (nroles > 0 && within_cap && less_imbalanced(l_scope, l_role)) {
      owner.swap(o_scope);
      load.swap(l_scope);
      chosen = MO_PLAN_SCOPE_GREEDY;
    } else {
      owner.swap(o_role);
      load.swap(l_role);
      chosen = MO_PLAN_ROLE_GREEDY;
    }
  }
  for (int32_t i = 0; i < nroles; ++i) owner_out[i] = owner[size_t(i)];
  if (load_out)
    for (int32_t r = 0; r < world; ++r) load_out[r] = load[size_t(r)];
  if (chosen_out) *chosen_out = chosen;
  return MO_OK;
}
