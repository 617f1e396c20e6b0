"""GPU parity of tk_decode_stream with the oracle's streaming decoder: the
page's worked example, random chunkings of multilingual text, trailing
partial characters flushed at the end, and errors that leave the state as
it was."""
import json
import os

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "stream_decode.json")


def test_page_example_hindi_token_boundary():
    import byte_level_bpe_gb300 as tk
    g = json.load(open(GOLDEN))
    toks = [bytes.fromhex(h) for h in g["tokens_hex"]]
    table = [bytes([i]) for i in range(256)] + [t for t in toks if len(t) > 1]
    gpu = tk.Tokenizer(table, {}, max_bytes=1 << 12, max_segments=4)
    ids = [table.index(t) for t in toks]
    dec = gpu.stream_decoder()
    assert [dec.feed([i]).hex() for i in ids] == g["emits_hex"]
    assert dec.finish().hex() == g["final_hex"]
    gpu.close()


def test_random_chunkings_match_oracle(full_table):
    import byte_level_bpe_gb300 as tk
    ranks = [(t, i) for i, t in enumerate(full_table)] + workloads.multilingual_table(full_table)
    enc = oracle.Encoding(ranks, {})
    gpu = tk.Tokenizer(ranks, {}, max_bytes=1 << 20, max_segments=4)
    text = workloads.multilingual_text(full_table, n_bytes=200000, seed=11)
    text = text.tobytes() if isinstance(text, np.ndarray) else bytes(text)
    ids = enc.encode(text)
    rng = np.random.default_rng(5)
    for trial in range(4):
        k = [60, 400, 2000, 8][trial]
        cuts = np.sort(rng.choice(np.arange(0, len(ids) + 1), size=k, replace=True))
        o_dec, g_dec = oracle.StreamDecoder(enc), gpu.stream_decoder()
        got = []
        for a, b in zip(np.r_[0, cuts], np.r_[cuts, len(ids)]):
            e_o = o_dec.feed(ids[a:b])
            e_g = g_dec.feed(ids[a:b])
            assert e_g == e_o, (trial, a, b)
            got.append(e_g)
        assert g_dec.finish() == o_dec.finish()
        assert b"".join(got) == text
    gpu.close()


def test_trailing_partial_character_is_flushed_at_the_end():
    import byte_level_bpe_gb300 as tk
    # tokens that end inside a character: an emoji cut after 2 and 3 bytes
    emoji = "\U0001F600".encode()
    table = [bytes([i]) for i in range(256)] + [b"a" + emoji[:2], emoji[2:], b"z" + emoji[:3]]
    enc = oracle.Encoding(table, {})
    gpu = tk.Tokenizer(table, {}, max_bytes=1 << 12, max_segments=4)
    for seq in ([256], [256, 257], [256, 257, 0x80], [258], [258, 0x41], [258, emoji[3]], [0xF0],
                [0xF0, 0x9F, 0x98], [0xED, 0xA0], [0xE0, 0x80]):
        o_dec, g_dec = oracle.StreamDecoder(enc), gpu.stream_decoder()
        outs_o = [o_dec.feed([i]) for i in seq] + [o_dec.finish()]
        outs_g = [g_dec.feed([i]) for i in seq] + [g_dec.finish()]
        assert outs_g == outs_o, seq
        assert b"".join(outs_g) == enc.decode(seq)
    gpu.close()


def test_errors_leave_the_state_unchanged(full_table):
    import byte_level_bpe_gb300 as tk
    from byte_level_bpe_gb300 import native
    gpu = tk.Tokenizer(full_table, workloads.SPECIALS, max_bytes=1 << 12, max_segments=4)
    st = torch.cuda.current_stream().cuda_stream
    state = native.DecodeState()
    # hold back the first two bytes of an emoji (bytes are their own ids)
    ids = torch.tensor([0xF0, 0x9F], dtype=torch.int32, device="cuda")
    out = torch.empty(16, dtype=torch.uint8, device="cuda")
    rc, m = native.tk_decode_stream(gpu.handle, gpu.workspace, state, ids.data_ptr(), 2, 0,
                                    out.data_ptr(), out.numel(), st)
    assert rc == 0 and m == 0 and state.n_pending == 2
    # too small an output: the required total comes back, the state stays
    rest = torch.tensor([0x98, 0x80, 65], dtype=torch.int32, device="cuda")
    rc, m = native.tk_decode_stream(gpu.handle, gpu.workspace, state, rest.data_ptr(), 3, 0,
                                    out.data_ptr(), 3, st, raise_on_error=False)
    assert rc == native.TK_E_CAPACITY and m == 5 and state.n_pending == 2
    # an unknown id: the state stays too
    bad = torch.tensor([0x98, 100256], dtype=torch.int32, device="cuda")
    rc, _ = native.tk_decode_stream(gpu.handle, gpu.workspace, state, bad.data_ptr(), 2, 0,
                                    out.data_ptr(), out.numel(), st, raise_on_error=False)
    assert rc == native.TK_E_BADID and state.n_pending == 2
    rc, m = native.tk_decode_stream(gpu.handle, gpu.workspace, state, rest.data_ptr(), 3, 1,
                                    out.data_ptr(), out.numel(), st)
    assert rc == 0 and out[:m].cpu().numpy().tobytes() == "\U0001F600A".encode()
    assert state.n_pending == 0
    gpu.close()


def test_decode_segments_matches_oracle(full_table, full_enc):
    import byte_level_bpe_gb300 as tk
    from byte_level_bpe_gb300 import native
    segs = workloads.agentic_segments(full_table, seed=7, scale=0.01)
    ids, off = full_enc.encode_segments(segs, tiktoken_safe=True)
    gpu = tk.Tokenizer(full_table, workloads.SPECIALS, max_bytes=1 << 20, max_segments=len(segs) + 1)
    d_ids = torch.from_numpy(np.ascontiguousarray(ids, np.int32)).cuda()
    d_off = torch.from_numpy(np.ascontiguousarray(off, np.int64)).cuda()
    out, boff = gpu.decode_segments(d_ids, d_off)
    parts = [full_enc.decode(ids[off[s]:off[s + 1]]) for s in range(len(segs))]
    assert out.cpu().numpy().tobytes() == b"".join(parts)
    assert boff.cpu().numpy().tolist() == np.r_[0, np.cumsum([len(p) for p in parts])].tolist()
    text, seg_off, _ = workloads.pack_segments(segs)
    assert out.cpu().numpy().tobytes() == text.tobytes()          # round trip of the encode
    assert boff.cpu().numpy().tolist() == seg_off.tolist()
    # offsets that do not run from 0 to n are refused
    bad = d_off.clone()
    bad[1] = bad[2] + 1
    rc, _ = native.tk_decode_segments(gpu.handle, gpu.workspace, d_ids.data_ptr(), len(ids), bad.data_ptr(),
                                      len(segs), out.data_ptr(), out.numel(),
                                      torch.empty(len(segs) + 1, dtype=torch.int64, device="cuda").data_ptr(),
                                      torch.cuda.current_stream().cuda_stream, raise_on_error=False)
    assert rc == native.TK_E_ARG
    gpu.close()
