"""Plain, slow, fp64 CPU oracle for retrieve + Chunked RoPE + paged KV injection.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product (the
``kv_cache_injection_gb300`` package and its CUDA library) never imports, calls
or links it, and this package imports nothing from the product: the two share
no code.  Inputs reach both sides from the seeded generators in ``synth``.

What it computes follows "InferScale: GPU-Native KV Injection for Personalized
LLM Serving" (arXiv 2607.27090), as summarised on the pages:

* retrieval of the k relevant facts from a GPU-resident store of semantic
  embeddings (abstract; "Conception de Système Native au GPU"), read as exact
  cosine similarity followed by top-k (``retrieval``);
* Chunked RoPE: keys are stored before rotation and rotated to their serving
  positions once the retrieved facts are composed into one contiguous segment
  ("Méthodologie", phase 2, "Stockage Pré-RoPE" / "Rotation Dynamique"),
  exact by Theorem 6 (``rope``);
* the scatter-copy of the composed K/V into a vLLM-style paged KV cache
  ("Méthodologie", phase 2, "Injection") (``inject``);
* Theorem 3 / Theorem 6 self-checks on a tiny one-layer causal attention
  (``attention``);
* Context-Window Encoding ("Méthodologie", phase 1): each fact encoded with a
  window of w preceding turns, only the fact's pre-RoPE K/V kept (``cwe``),
  on a tiny multi-layer decoder with synthetic weights (``model``);
* storage encodings, including the FP8 E4M3 cache (``numerics``).

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
hand-computed values, invariants and brute force; none is "parity unpinned".
"""
