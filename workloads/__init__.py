"""Seeded synthetic inputs for byte-level BPE encoding.

This module only draws random numbers and lays out bytes. It holds none of the
encoder's arithmetic (no split, no merge, no chunking), so both the CPU oracle's
tests and the CUDA path's tests and benchmark can use it.

Workloads (sizes and mixes stand in for the pages' corpora, which are not
available; see the design notes for the full recipe):
  tiny      64 KiB of Zipf(1.1) lowercase words for the 4,096-merge trained table
  full      1 MiB of prose over a 100,256-rank synthetic table
  agentic   ~4 M characters in 2,000 typed segments with safe chunking
  multiling 8 MiB of ASCII / CJK / Devanagari / emoji / control bytes
  serving   4,096 requests, 256 MiB, 90% of each repeating an earlier request
"""
from .gen import (  # noqa: F401
    SPECIALS,
    agentic_segments,
    full_table,
    multilingual_table,
    multilingual_text,
    prose_text,
    serving_batch,
    tiny_corpus,
    tiny_input,
    pack_segments,
    input_sha256,
    table_sha256,
    manifest_inputs,
)
