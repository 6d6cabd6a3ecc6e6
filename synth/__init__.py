"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This package generates *inputs only*: fact lengths, embeddings, query
embeddings, per-fact pre-RoPE keys and raw values, segment start positions
and block tables.  It contains none of the method's arithmetic (no cosine
similarity, no top-k, no rotary embedding, no slot mapping).

Keys and values are produced by a counter-based generator (SplitMix64 words,
Irwin-Hall sum of twelve 16-bit uniforms) that has two implementations built
from the same published definition: ``synth.kvgen`` (numpy, host) and
``synth/csrc/synthgen.cu`` (CUDA, device).  Both give identical bits, so the
device can fill a store of ~100 GB while the host oracle regenerates only the
facts it needs.
"""
