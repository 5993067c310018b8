"""Greedy draft acceptance for one MTP verify batch.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"Support Step3.5/3.7 flash mtp3" (llama.cpp PR #24340), "Overview" data-flow
trace, Round 1: the target batch is [id_last, d1, d2, d3] with logits for every
row (step 1); verify samples each row of the target's logits and compares row
i with draft i+1, stopping at the first mismatch, where the target's token is
taken instead (step 4); accept then keeps the matched drafts plus that token,
and the hidden state handed to the next round is verify_h[n_accepted]
(step 5).  Greedy sampling (temperature 0, as in the PR's runs) is argmax;
ties go to the lowest token id.
"""

import numpy as np


def argmax_lowest(row):
    """Index of the largest value; the first (lowest) index on ties."""
    row = np.asarray(row)
    return int(np.flatnonzero(row == row.max())[0])


def greedy_accept(draft_ids, logits):
    """draft_ids [k], logits [k+1, V] -> (n_accepted, next_token, argmaxes).

    n_accepted is the largest n <= k with argmax(row i) == draft[i] for all
    i < n; next_token = argmax(row n_accepted) (the correction token, or the
    bonus token when every draft matched).
    """
    draft_ids = [int(d) for d in draft_ids]
    k = len(draft_ids)
    logits = np.asarray(logits)
    assert logits.shape[0] == k + 1
    a = [argmax_lowest(logits[i]) for i in range(k + 1)]
    n = 0
    while n < k and a[n] == draft_ids[n]:
        n += 1
    return n, a[n], a
