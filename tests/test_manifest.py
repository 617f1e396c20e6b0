"""The seeded generators reproduce the inputs recorded in workloads/manifest.json
(written by workloads/write_manifest.py): every workload input and the two
generated tables hash to the recorded sha256."""
import json
import os

import numpy as np

import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_generated_inputs_match_manifest():
    with open(os.path.join(ROOT, "workloads", "manifest.json")) as f:
        m = json.load(f)
    got = workloads.manifest_inputs()
    assert set(got) == set(m["inputs"])
    for name, (text, off, allow) in got.items():
        rec = m["inputs"][name]
        assert workloads.input_sha256(text, off, allow) == rec["sha256"], name
        assert text.size == rec["bytes"] and len(off) - 1 == rec["segments"], name
    table = workloads.full_table()
    assert workloads.table_sha256(table) == m["tables"]["full"]["sha256"]
    ext = workloads.multilingual_table(table)
    assert workloads.table_sha256(ext) == m["tables"]["multilingual_extension"]["sha256"]
    corpus = np.frombuffer(workloads.tiny_corpus(), np.uint8)
    assert workloads.input_sha256(corpus, [0], [0]) == m["tables"]["corpus_tiny_sha256"]
