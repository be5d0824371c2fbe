"""Confidence-gated prefetch rule (oracle; test infrastructure only).

"Paging the Experts" §3.3: during prefill, the prefetcher takes the
preceding step's highest-weight expert of the same layer and prefetches it
when its normalised weight reaches 0.20; the actual routing and arithmetic
do not change. §5.2 counts the loads as useful or wasted (6,223 and 4,111 of
10,334 at 512 MiB).

Reading for steps of several tokens, which the page (serial single-token
prefill) leaves open: the step's last token is the one that precedes the
next step, so its rank-0 expert (the highest weight of its selection, the
first entry of its top-k) and that expert's combine weight make the
prediction for the next step of the layer. With one token per step this is
exactly the page's rule.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

THRESHOLD = 0.20


def prediction(idx: np.ndarray, weights: np.ndarray, threshold: float = THRESHOLD) -> Optional[int]:
    """idx int [T, k] (descending weight), weights [T, k]: the expert to
    prefetch for the layer's next step, or None when the last token's top
    weight is below the threshold."""
    if idx.shape[0] == 0:
        return None
    e, w = int(idx[-1, 0]), float(weights[-1, 0])
    return e if w >= threshold else None
