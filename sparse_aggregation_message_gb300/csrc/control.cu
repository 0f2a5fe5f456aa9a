// Epoch-level adaptive control of the SYLVIE guide, sections 8, 10 and 11:
// the Coordinator's averaged and smoothed loss, the loss-descent rate (LDR),
// the Quant Orchestrator's base width and the Pipeline Adaptor's choice of
// synchronous or asynchronous execution for the next epoch.  Host code only.
//
// Reading of the sign: the pages define LDR_t = (F_t - F_{t-1}) / et_t but
// describe a smaller LDR as worse progress (and double the width / force a
// synchronous epoch on it).  Both statements hold when LDR is the descent
// rate (F_{t-1} - F_t) / et_t, which is what is computed here.
#include "internal.h"

using namespace gnn;

static bool is_width(int b) { return b == 1 || b == 2 || b == 4 || b == 8; }

extern "C" gnn_status gnn_ldr_init(gnn_ldr_state* st, double lambda, int32_t delta,
                                   int32_t b_min, int32_t b_max) {
  GNN_REQUIRE(st, "gnn_ldr_init: NULL state");
  GNN_REQUIRE(lambda >= 0.0 && lambda < 1.0, "gnn_ldr_init: lambda must be in [0, 1)");
  GNN_REQUIRE(delta >= 1 && delta <= GNN_LDR_MAX_DELTA, "gnn_ldr_init: delta must be 1..%d",
              GNN_LDR_MAX_DELTA);
  GNN_REQUIRE(is_width(b_min) && is_width(b_max) && b_min <= b_max,
              "gnn_ldr_init: b_min <= b_max, both in {1, 2, 4, 8}");
  st->lambda = lambda;
  st->delta = delta;
  st->b_min = b_min;
  st->b_max = b_max;
  st->t = 0;
  st->base_bits = b_min;
  st->async_next = 0;
  st->F = 0.0;
  for (int i = 0; i <= GNN_LDR_MAX_DELTA; ++i) st->ldr[i] = 0.0;
  return GNN_OK;
}

extern "C" gnn_status gnn_ldr_update(gnn_ldr_state* st, const double* partition_loss,
                                     int32_t n_parts, double epoch_seconds) {
  GNN_REQUIRE(st && partition_loss && n_parts >= 1, "gnn_ldr_update: bad arguments");
  GNN_REQUIRE(epoch_seconds > 0.0, "gnn_ldr_update: epoch time must be positive");
  GNN_REQUIRE(st->delta >= 1 && st->delta <= GNN_LDR_MAX_DELTA, "gnn_ldr_update: state not initialised");
  // Coordinator: L_t = mean of the partitions' losses, F_t = lambda F_{t-1} + (1-lambda) L_t
  double sum = 0.0;
  for (int i = 0; i < n_parts; ++i) sum += partition_loss[i];
  const double L = sum / (double)n_parts;
  const int t = st->t;
  double F, ldr;
  if (t == 0) {  // the first epoch initialises the smoothed loss
    F = L;
    ldr = 0.0;
  } else {
    const double a = st->lambda * st->F;
    const double b = (1.0 - st->lambda) * L;
    F = a + b;
    ldr = (st->F - F) / epoch_seconds;
  }
  const int ring = st->delta + 1;
  st->ldr[t % ring] = ldr;
  if (t == 0) {
    st->base_bits = st->b_min;
  } else if (t > st->delta) {
    const double past = st->ldr[(t - st->delta) % ring];
    if (ldr < past) {  // descent slowed: more precision, synchronous refresh
      st->base_bits = st->base_bits * 2 > st->b_max ? st->b_max : st->base_bits * 2;
      st->async_next = 0;
    } else {  // not worse: fewer bits, asynchronous pipeline
      st->base_bits = st->base_bits / 2 < st->b_min ? st->b_min : st->base_bits / 2;
      st->async_next = 1;
    }
  }
  st->F = F;
  st->t = t + 1;
  return GNN_OK;
}
