"""Exact cosine top-k retrieval over one user's facts, in fp64.

The pages say InferScale keeps a semantic embedding beside each fact's KV on the
GPU and retrieves the relevant facts at serving time under a budget k
(abstract; "Problématique": subset of k facts; "Conception de Système Native au
GPU": GPU-resident semantic retrieval).  The index they name is not described,
so retrieval here is the plain definition: the cosine similarity of the query
with every stored embedding of the query's user, then the k best.

Readings where the pages are silent:
* ties in score go to the lower fact id;
* the result is ordered by descending score (then ascending id);
* a user with fewer than k facts returns all of them;
* the cosine with a zero vector is taken as 0.
"""
from __future__ import annotations

import numpy as np


def cosine_scores(query: np.ndarray, embeddings: np.ndarray) -> np.ndarray:
    """s_j = <q, e_j> / (|q| |e_j|) in fp64 from the stored values."""
    q = np.asarray(query, dtype=np.float64)
    X = np.asarray(embeddings, dtype=np.float64)
    dots = X @ q
    denom = np.linalg.norm(X, axis=1) * np.linalg.norm(q)
    out = np.zeros(X.shape[0], dtype=np.float64)
    nz = denom > 0
    out[nz] = dots[nz] / denom[nz]
    return out


def topk(scores: np.ndarray, fact_ids: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray]:
    """The min(k, n) entries with the largest score, ties to the lower id,
    ordered by (descending score, ascending id)."""
    scores = np.asarray(scores, dtype=np.float64)
    fact_ids = np.asarray(fact_ids, dtype=np.int64)
    order = np.lexsort((fact_ids, -scores))
    sel = order[:min(k, len(order))]
    return fact_ids[sel], scores[sel]


def retrieve(query: np.ndarray, user_embeddings: np.ndarray, user_fact_ids: np.ndarray,
             k: int) -> tuple[np.ndarray, np.ndarray]:
    return topk(cosine_scores(query, user_embeddings), user_fact_ids, k)
