// host_budget.cu -- the adaptive draft-tree budget of a serving loop (host code only:
// no device memory, no stream, no kernel).
//
// "Thinking Budget 与 EAGLE-3", 服务端应怎样联合控制: the execution controller changes
// only the speculative budget, never the target's decoding.  It lowers the draft
// tree budget when the recent accepted length is low or drafting is costly, raises
// it cautiously when acceptance is stable and verification has spare capacity, and
// keeps every change within bounds, behind a cool-down window, with a fallback
// baseline, so that short-term noise does not make it oscillate.  The budget is a
// ladder of tree shapes (node budget N, depth D), cheapest first ("论文专题讲解：
// EAGLE-3", Draft tree 配置: the tree is a budget of nodes and a depth).
//
// Per request the controller keeps a running mean of the accepted length (drafted
// tokens accepted per round) and a running mean absolute deviation from it, both
// exponentially weighted; a level may change only after `warmup` rounds at it and
// not while a cool-down is running.
#include <math.h>
#include <stdint.h>

#include "e3_common.cuh"

using namespace e3;

namespace {

e3_status check_policy(const e3_budget_policy* p, const char* fn) {
  E3_REQUIRE(p != nullptr, E3_ERR_INVALID_ARG, "%s: null policy", fn);
  E3_REQUIRE(p->n_levels >= 1 && p->n_levels <= E3_MAX_BUDGET_LEVELS, E3_ERR_SHAPE, "%s: n_levels %d not in [1, %d]",
             fn, p->n_levels, E3_MAX_BUDGET_LEVELS);
  for (int i = 0; i < p->n_levels; ++i) {
    E3_REQUIRE(p->nodes[i] >= 1 && p->depth[i] >= 1 && p->depth[i] <= p->nodes[i], E3_ERR_SHAPE,
               "%s: level %d has nodes %d, depth %d", fn, i, p->nodes[i], p->depth[i]);
    if (i > 0)
      E3_REQUIRE(p->nodes[i] >= p->nodes[i - 1] && p->depth[i] >= p->depth[i - 1], E3_ERR_SHAPE,
                 "%s: levels must not get cheaper (level %d)", fn, i);
  }
  E3_REQUIRE(p->min_level >= 0 && p->min_level <= p->max_level && p->max_level < p->n_levels, E3_ERR_SHAPE,
             "%s: bounds [%d, %d] outside the %d levels", fn, p->min_level, p->max_level, p->n_levels);
  E3_REQUIRE(p->base_level >= p->min_level && p->base_level <= p->max_level, E3_ERR_SHAPE,
             "%s: base level %d outside the bounds", fn, p->base_level);
  E3_REQUIRE(p->alpha > 0.0f && p->alpha <= 1.0f, E3_ERR_INVALID_ARG, "%s: alpha must be in (0, 1]", fn);
  E3_REQUIRE(p->low >= 0.0f && p->low <= p->high && p->high <= 1.0f, E3_ERR_INVALID_ARG,
             "%s: need 0 <= low <= high <= 1", fn);
  E3_REQUIRE(p->spread >= 0.0f && p->min_spare >= 0.0f && p->max_draft_cost > 0.0f, E3_ERR_INVALID_ARG,
             "%s: spread, min_spare must be >= 0 and max_draft_cost > 0", fn);
  E3_REQUIRE(p->cooldown >= 0 && p->warmup >= 1, E3_ERR_INVALID_ARG, "%s: cooldown >= 0 and warmup >= 1", fn);
  return E3_OK;
}

void reset(const e3_budget_policy* p, e3_budget_state* s) {
  s->level = p->base_level;
  s->hold = 0;
  s->rounds = 0;
  // a fresh request starts from the baseline's midpoint between the two thresholds
  s->mean = 0.5f * (p->low + p->high) * static_cast<float>(p->depth[p->base_level]);
  s->dev = 0.0f;
}

}  // namespace

extern "C" {

E3_API e3_status eagle3_budget_init(const e3_budget_policy* pol, e3_budget_state* st, int B) {
  clear_error();
  const e3_status ps = check_policy(pol, "eagle3_budget_init");
  if (ps != E3_OK) return ps;
  E3_REQUIRE(st != nullptr && B >= 1, E3_ERR_INVALID_ARG, "eagle3_budget_init: null state or B < 1");
  for (int b = 0; b < B; ++b) reset(pol, &st[b]);
  return E3_OK;
}

E3_API e3_status eagle3_budget_update(const e3_budget_policy* pol, e3_budget_state* st, int B, const int32_t* acc_len,
                                      float spare, float draft_cost, int32_t* level) {
  clear_error();
  const e3_status ps = check_policy(pol, "eagle3_budget_update");
  if (ps != E3_OK) return ps;
  E3_REQUIRE(st != nullptr && acc_len != nullptr && level != nullptr && B >= 1, E3_ERR_INVALID_ARG,
             "eagle3_budget_update: null pointer or B < 1");
  E3_REQUIRE(isfinite(spare) && isfinite(draft_cost), E3_ERR_INVALID_ARG,
             "eagle3_budget_update: spare and draft_cost must be finite");
  const bool costly = draft_cost > pol->max_draft_cost;
  const bool room = spare >= pol->min_spare;
  for (int b = 0; b < B; ++b) {
    e3_budget_state* s = &st[b];
    if (s->level < pol->min_level || s->level > pol->max_level || s->hold < 0 || s->rounds < 0 ||
        !isfinite(s->mean) || !isfinite(s->dev)) {
      reset(pol, s);  // a corrupt or out-of-bounds state falls back to the baseline
    }
    const int a = acc_len[b];
    if (a < 0 || a > pol->depth[s->level]) {  // no valid observation: back to the baseline
      reset(pol, s);
      level[b] = s->level;
      continue;
    }
    const float x = static_cast<float>(a);
    const float err = fabsf(x - s->mean);
    s->mean += pol->alpha * (x - s->mean);
    s->dev += pol->alpha * (err - s->dev);
    s->rounds += 1;
    if (s->hold > 0) {
      s->hold -= 1;
    } else if (s->rounds >= pol->warmup) {
      const float D = static_cast<float>(pol->depth[s->level]);
      const bool low = s->mean < pol->low * D;
      const bool stable_high = s->mean >= pol->high * D && s->dev <= pol->spread * D;
      int next = s->level;
      if ((low || costly) && s->level > pol->min_level) {
        next = s->level - 1;
      } else if (stable_high && room && !costly && s->level < pol->max_level) {
        next = s->level + 1;
      }
      if (next != s->level) {
        s->level = next;
        s->hold = pol->cooldown;
        s->rounds = 0;
      }
    }
    level[b] = s->level;
  }
  return E3_OK;
}

}  // extern "C"
