// Training-free layer selection: the greedy search for the F/S pattern.
//
// notes page ("NLP--IndexCache"), section "核心算法：Greedy Layer Selection",
// and deep-read page ("IndexCache：跨层复用稀疏注意力的索引"), section
// "Training-free：直接用语言模型损失选择 Full 层":
//   start from all-Full; layer 0 is never a candidate; in each of K rounds,
//   turn every remaining Full layer (except 0) into Shared on trial, evaluate
//   the model's loss under that pattern, and commit the flip whose loss is
//   lowest.  K rounds cost sum_{i<K} (N - 1 - i) = K(N-1) - K(K-1)/2 loss
//   evaluations (full forwards).
//
// The loss is the caller's: a callback that runs whatever model and
// calibration data it owns under the proposed pattern.  Ties in loss go to
// the lower layer index (the deep-read page's search takes the minimum of
// (loss, layer) pairs).  Host code only.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <string>
#include <vector>

#include "ic_common.cuh"
#include "ic_kernels.h"

extern "C" __attribute__((visibility("default"))) ic_status ic_greedy_full_layers(
    int n_layers, int removals, ic_loss_fn evaluate_loss, void* user, char* pattern_out, long long* forwards_out) {
  ic::clear_error();
  if (forwards_out) *forwards_out = 0;
  if (n_layers < 1) return ic::report_error(IC_ERR_ARG, "n_layers must be >= 1");
  if (removals < 0 || removals > n_layers - 1)
    return ic::report_error(IC_ERR_ARG, "removals must lie in [0, n_layers - 1]: layer 0 always stays Full");
  if (!evaluate_loss || !pattern_out) return ic::report_error(IC_ERR_ARG, "null callback or output pointer");
  std::string roles(static_cast<size_t>(n_layers), 'F');
  std::vector<int> remaining;
  for (int l = 1; l < n_layers; ++l) remaining.push_back(l);
  long long forwards = 0;
  for (int step = 0; step < removals; ++step) {
    double best_loss = 0.0;
    int best_at = -1;   // position in `remaining`
    for (size_t i = 0; i < remaining.size(); ++i) {
      std::string trial = roles;
      trial[static_cast<size_t>(remaining[i])] = 'S';
      const double loss = evaluate_loss(trial.c_str(), user);
      ++forwards;
      if (forwards_out) *forwards_out = forwards;
      if (isnan(loss)) {
        memcpy(pattern_out, roles.c_str(), roles.size() + 1);
        char msg[160];
        snprintf(msg, sizeof(msg),
                 "the loss callback returned NaN for a trial that makes layer %d Shared (removal step %d)",
                 remaining[i], step);
        return ic::report_error(IC_ERR_ARG, msg);
      }
      // `remaining` is ascending, so a strict < keeps the lower layer on a tie
      if (best_at < 0 || loss < best_loss) {
        best_loss = loss;
        best_at = static_cast<int>(i);
      }
    }
    roles[static_cast<size_t>(remaining[static_cast<size_t>(best_at)])] = 'S';
    remaining.erase(remaining.begin() + best_at);
  }
  memcpy(pattern_out, roles.c_str(), roles.size() + 1);
  return IC_OK;
}
