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
reading of it, with every step a plain definition (in "bf16" activation mode
the MoE layers' inputs are additionally rounded to bf16, as a bf16 layer
takes them):
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
  draft cut   ("Step-3.5-Flash MTP GGUF", "Usage" and "Notes": the server flag
              --spec-draft-p-min, 0.65 recommended; "Support Step3.5/3.7 flash
              mtp3", test settings: 0.0 in the PR's runs.  The pages give the
              flag and its values only; the reading here is the plain one:)
              draft j's confidence is the probability of its token under the
              draft logits, p_j = max_v softmax(draft_logits[j])_v =
              1 / sum_v exp(l_v - max l); drafting stops at the first j with
              p_j < p_min, and that draft and every later one are dropped
              (reported as -1).  p_min = 0 keeps every draft.
  acceptance  greedy: oracle.accept.greedy_accept(kept drafts, logits of the
              kept drafts' verify rows)
Since drafts are a function of the target's hidden states here, the target
runs first; the work of the round and the acceptance rule are those of the
trace.
"""

import numpy as np

from . import accept, moe

F64 = np.float64


def round_bf16(x):
    """Round to the nearest bf16 value (8 significant bits, ties to even),
    directly from fp64; values stay fp64 arrays."""
    x = np.asarray(x, F64)
    m, e = np.frexp(x)                  # x = m 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.round(np.ldexp(m, 8)), e - 8)  # np.round: halves to even


def rmsnorm(x, eps=1e-6):
    """Row-wise v / sqrt(mean(v^2) + eps), weight 1, fp64."""
    x = np.asarray(x, F64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def lm_logits(h, lm: moe.QTensor, eps=1e-6):
    """logits [T, V] = W_lm . rmsnorm(h) for h [T, H]."""
    return rmsnorm(h, eps) @ lm.dense().T


def target_stack(x, layers, eps=1e-6, routes=None, layer_forward=None, act="f64"):
    """h_tgt for the verify batch x [T, H] through pre-norm residual MoE layers.
    If `routes` is a list, each layer's routing dict is appended to it.
    ``layer_forward(x, L)``, if given, stands in for ``moe.forward(x, L)``.
    act = "bf16": the layers' inputs are bf16 values (rmsnorm(h) rounded to
    nearest even); their outputs and the residual stream keep full precision."""
    fwd = moe.forward if layer_forward is None else layer_forward
    io = round_bf16 if act == "bf16" else (lambda v: v)
    h = np.asarray(x, F64)
    for L in layers:
        y, r = fwd(io(rmsnorm(h, eps)), L)
        if routes is not None:
            routes.append(r)
        h = h + y
    return h


def draft_probability(row):
    """The largest softmax probability of a logit row, 1 / sum_v exp(l_v - max l),
    in fp64."""
    row = np.asarray(row, F64)
    return float(1.0 / np.exp(row - row.max()).sum())


def cut_drafts(drafts, probs, p_min):
    """The drafts kept under the confidence cut: the longest prefix whose
    probabilities are all >= p_min.  Returns (kept drafts, n_drafted)."""
    n = 0
    while n < len(drafts) and probs[n] >= p_min:
        n += 1
    return list(drafts[:n]), n


def mtp_round(x, layers, heads, lm: moe.QTensor, noise, eps=1e-6, p_min=0.0, layer_forward=None, act="f64"):
    """One round.  x [k+1, H]; heads: k layers; noise [k][k][H] (head j uses
    rows 0..j of noise[j]); p_min the draft confidence cut.  Returns a dict
    with h_tgt, logits, head_out (list of [j+1, H]), draft_rows [k, H],
    draft_logits [k, V], draft_probs [k], drafts [k] (-1 past the cut),
    n_drafted, n_accepted, next_token, argmax (the target's per-row argmax)
    and the routing dicts of every target layer (target_routes) and head
    (head_routes).  ``layer_forward(x, L)``, if given, stands in for
    ``moe.forward(x, L)``.  act = "bf16": every MoE layer's (and head's)
    input is a bf16 value (see target_stack); outputs, the residual stream,
    the draft rows and the logits keep full precision."""
    fwd = moe.forward if layer_forward is None else layer_forward
    io = round_bf16 if act == "bf16" else (lambda v: v)
    k = len(heads)
    x = np.asarray(x, F64)
    assert x.shape[0] == k + 1
    target_routes, head_routes = [], []
    h_tgt = target_stack(x, layers, eps, target_routes, layer_forward=fwd, act=act)
    logits = lm_logits(h_tgt, lm, eps)
    head_out, rows = [], []
    for j, head in enumerate(heads):
        ht = h_tgt[: j + 1] + np.asarray(noise[j][: j + 1], F64)
        y, hr = fwd(io(rmsnorm(ht, eps)), head)
        head_routes.append(hr)
        head_out.append(y)
        rows.append(ht[j])
    rows = np.stack(rows) if rows else np.zeros((0, x.shape[1]))
    draft_logits = lm_logits(rows, lm, eps)
    tokens = [accept.argmax_lowest(r) for r in draft_logits]
    probs = [draft_probability(r) for r in draft_logits]
    kept, n_drafted = cut_drafts(tokens, probs, p_min)
    n, nxt, _ = accept.greedy_accept(kept, logits[: n_drafted + 1])
    amax = [accept.argmax_lowest(r) for r in logits]
    drafts = kept + [-1] * (k - n_drafted)
    return dict(h_tgt=h_tgt, logits=logits, head_out=head_out, draft_rows=rows,
                draft_logits=draft_logits, draft_probs=probs, drafts=drafts, n_drafted=n_drafted,
                n_accepted=n, next_token=nxt, argmax=amax, target_routes=target_routes,
                head_routes=head_routes)
