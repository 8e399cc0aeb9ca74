"""The same iteration run one request at a time (oracle).

[houmin] 3.1.2 "方案" and [arcsin2] §3.2: selective batching is exact -- the
token-wise operations do not mix rows of different requests and attention is
computed per request -- so executing the batch one request at a time must
give every request the same result.  ``recompute`` also checks the K/V cache
itself: the logits of a request after an increment equal those of one
initiation pass over its whole token sequence.
"""

from __future__ import annotations

from typing import List, Sequence

import numpy as np

from . import model
from .model import BatchItem, KVStore, Result


def iteration(w: dict, n_heads: int, batch: Sequence[BatchItem], store: KVStore) -> Result:
    hid, log, nxt = [], [], []
    for it in batch:
        r = model.iteration(w, n_heads, [it], store)
        hid.append(r.hidden[0])
        log.append(r.logits[0])
        nxt.append(r.next_tokens[0])
    return Result(np.stack(hid), np.stack(log), nxt)


def recompute(w: dict, n_heads: int, sequence: List[int]) -> Result:
    """Initiation pass over ``sequence`` with an empty cache (no reuse)."""
    store = KVStore(len(w["layers"]), w["tok_emb"].shape[1])
    return model.iteration(w, n_heads, [BatchItem(-1, list(sequence), 0)], store)
