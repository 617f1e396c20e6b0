"""Writes workloads/manifest.json: the sha256 of every generated input and of
the generated tables (run once after a change to the generators):

    python workloads/write_manifest.py

The inputs are regenerated from their seeds wherever they are used (nothing
large is committed); the manifest lets tests and the benchmark check that what
they generated is what was recorded. The tiny table is trained from the tiny
corpus by the oracle's trainer at test time and is not recorded here.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import workloads  # noqa: E402


def main():
    table = workloads.full_table()
    m = {"inputs": {}, "tables": {}}
    for name, (text, off, allow) in workloads.manifest_inputs().items():
        m["inputs"][name] = {"sha256": workloads.input_sha256(text, off, allow),
                             "bytes": int(text.size), "segments": int(len(off) - 1)}
    m["tables"]["full"] = {"sha256": workloads.table_sha256(table), "tokens": len(table)}
    ext = workloads.multilingual_table(table)
    m["tables"]["multilingual_extension"] = {"sha256": workloads.table_sha256(ext), "tokens": len(ext)}
    m["tables"]["corpus_tiny_sha256"] = workloads.input_sha256(
        __import__("numpy").frombuffer(workloads.tiny_corpus(), "uint8"), [0], [0])
    with open(os.path.join(HERE, "manifest.json"), "w") as f:
        json.dump(m, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps(m, indent=1, sort_keys=True))


if __name__ == "__main__":
    main()
