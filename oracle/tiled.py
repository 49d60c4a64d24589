"""The pages' tiled online-softmax algorithm, restated in fp64 numpy.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  It exists so the tests can
check the method's exactness claim -- the tiled result equals the materialised
softmax result ("numerically identical", khetwal.com, "The Trick: Online
Softmax") -- for every block split, independently of the CUDA path.

Steps follow "FlashAttention (Conceptual)" in the worked example of
"FlashAttention: how a memory trick unlocked..." (khetwal.com), in its order:
outer loop over query blocks, inner loop over key/value blocks, per inner step
(1) score block, (2) new running max, (3) rescale the output block and the
normaliser, (4) block probabilities and their row sum, (5) update the
normaliser, (6) accumulate P V, (7) carry the max; then divide by the
normaliser.  Readings where the listing is silent or garbled:
  * the scores carry the scale factor (the score step in "The Quadratic Memory
    Bottleneck" is written with a scale);
  * the running max and normaliser are per query row ("for each row ... it
    maintains two values");
  * a block in which a row sees no key leaves that row's statistics unchanged
    (exp(-inf - -inf) is taken as a factor of 1 and the block's P as 0);
  * the log-sum-exp output is m + ln(normaliser).
"""
from __future__ import annotations

import numpy as np


def visible_mask(n, causal=False, kv_len=None, block_mask=None, tile=128):
    """Boolean [n, n] visibility: j < kv_len, j <= i if causal, tile bit set."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    vis = np.ones((n, n), dtype=bool)
    if kv_len is not None:
        vis &= j < int(kv_len)
    if causal:
        vis &= j <= i
    if block_mask is not None:
        bm = np.asarray(block_mask).astype(bool)
        vis &= bm[i // tile, j // tile]
    return vis


def tiled_attention(q, k, v, scale, block_q, block_k, *, causal=False, kv_len=None,
                    block_mask=None, tile=128):
    """One head, q/k/v [N, d].  Returns (O [N, d], LSE [N]) in float64."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n, d = q.shape
    vis = visible_mask(n, causal, kv_len, block_mask, tile)
    o = np.zeros((n, d))
    lse = np.empty(n)
    for i0 in range(0, n, block_q):
        i1 = min(i0 + block_q, n)
        q_block = q[i0:i1]
        o_block = np.zeros((i1 - i0, d))
        running_max = np.full(i1 - i0, -np.inf)
        running_normalizer = np.zeros(i1 - i0)
        for j0 in range(0, n, block_k):
            j1 = min(j0 + block_k, n)
            k_block, v_block = k[j0:j1], v[j0:j1]
            # 1. score block (masked entries are -inf)
            s_block = scale * (q_block @ k_block.T)
            s_block = np.where(vis[i0:i1, j0:j1], s_block, -np.inf)
            # 2. new running max
            local_max = s_block.max(axis=1)
            new_max = np.maximum(running_max, local_max)
            # 3. rescale the previous output and normaliser
            finite = np.isfinite(new_max)
            safe_max = np.where(finite, new_max, 0.0)
            factor = np.where(finite, np.exp(running_max - safe_max), 1.0)
            o_block *= factor[:, None]
            running_normalizer *= factor
            # 4. block probabilities and their row sum
            p_block = np.where(finite[:, None], np.exp(s_block - safe_max[:, None]), 0.0)
            local_normalizer = p_block.sum(axis=1)
            # 5. update the normaliser
            running_normalizer += local_normalizer
            # 6. accumulate this block's contribution
            o_block += p_block @ v_block
            # 7. carry the max
            running_max = new_max
        seen = running_normalizer > 0
        o[i0:i1] = np.where(seen[:, None], o_block / np.where(seen, running_normalizer, 1.0)[:, None], 0.0)
        lse[i0:i1] = np.where(seen, running_max + np.log(np.where(seen, running_normalizer, 1.0)), -np.inf)
    return o, lse
