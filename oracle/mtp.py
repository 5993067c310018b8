"""One synthetic MTP draft/verify round: target MoE stack, output norm, LM
head, draft heads and greedy acceptance, in fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"Support Step3.5/3.7 flash mtp3" (llama.cpp PR #24340), "Overview" data-flow
trace: a round drafts with three chained heads at batch sizes 1, 2, 3
(step 6), runs the target on [id_last, d1, d2, d3] with logits for every row
(steps 1-2), verifies row i against draft i+1 (step 4) and accepts (step 5);
h_tgt is the target hidden state before the output norm.  "Step-5 Preview
GGUF", "Precision distribution" table: the main output matrix is Q8_0.

The pages give the data flow but no synthetic model, so the round here is a
reading of it, with every step a plain definition:
  target      h_0 = x (the [k+1, H] verify batch); h_{l+1} = h_l +
              MoE_l(rmsnorm(h_l)) for the L target layers (pre-norm residual
              blocks: without the norm the SwiGLU, quadratic in its input,
              makes the synthetic stack's hidden state grow by orders of
              magnitude per layer); h_tgt = h_L
  logits      logits = W_lm . rmsnorm(h) with rmsnorm(v) = v / sqrt(mean(v^2) + eps)
              (weight 1), W_lm a Q8_0 matrix [V, H]
  drafts      head j (j = 0..k-1) is one MoE layer run on rmsnorm of the j+1
              rows h~_j = h_tgt[0..j] + noise[j][0..j] (the noise stands in
              for an imperfect draft model: it is what makes drafts differ from
              the target); its output is computed and compared as a layer output;
              draft token d_{j+1} = argmax W_lm . rmsnorm(h~_j[j])
  acceptance  greedy: oracle.accept.greedy_accept(d_1..d_k, logits)
Since drafts are a function of the target's hidden states here, the target
runs first; the work of the round and the acceptance rule are those of the
trace.
"""

import numpy as np

from . import accept, moe

F64 = np.float64


def rmsnorm(x, eps=1e-6):
    """Row-wise v / sqrt(mean(v^2) + eps), weight 1, fp64."""
    x = np.asarray(x, F64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def lm_logits(h, lm: moe.QTensor, eps=1e-6):
    """logits [T, V] = W_lm . rmsnorm(h) for h [T, H]."""
    return rmsnorm(h, eps) @ lm.dense().T


def target_stack(x, layers, eps=1e-6, routes=None):
    """h_tgt for the verify batch x [T, H] through pre-norm residual MoE layers.
    If `routes` is a list, each layer's routing dict is appended to it."""
    h = np.asarray(x, F64)
    for L in layers:
        y, r = moe.forward(rmsnorm(h, eps), L)
        if routes is not None:
            routes.append(r)
        h = h + y
    return h


def mtp_round(x, layers, heads, lm: moe.QTensor, noise, eps=1e-6):
    """One round.  x [k+1, H]; heads: k layers; noise [k][k][H] (head j uses
    rows 0..j of noise[j]).  Returns a dict with h_tgt, logits, head_out
    (list of [j+1, H]), draft_rows [k, H], draft_logits [k, V], drafts [k],
    n_accepted, next_token, argmax (the target's per-row argmax) and the routing
    dicts of every target layer (target_routes) and head (head_routes)."""
    k = len(heads)
    x = np.asarray(x, F64)
    assert x.shape[0] == k + 1
    target_routes, head_routes = [], []
    h_tgt = target_stack(x, layers, eps, target_routes)
    logits = lm_logits(h_tgt, lm, eps)
    head_out, rows = [], []
    for j, head in enumerate(heads):
        ht = h_tgt[: j + 1] + np.asarray(noise[j][: j + 1], F64)
        y, hr = moe.forward(rmsnorm(ht, eps), head)
        head_routes.append(hr)
        head_out.append(y)
        rows.append(ht[j])
    rows = np.stack(rows) if rows else np.zeros((0, x.shape[1]))
    draft_logits = lm_logits(rows, lm, eps)
    drafts = [accept.argmax_lowest(r) for r in draft_logits]
    n, nxt, amax = accept.greedy_accept(drafts, logits)
    return dict(h_tgt=h_tgt, logits=logits, head_out=head_out, draft_rows=rows,
                draft_logits=draft_logits, drafts=drafts, n_accepted=n, next_token=nxt,
                argmax=amax, target_routes=target_routes, head_routes=head_routes)
