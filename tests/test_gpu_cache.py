"""The cross-call word cache never changes a result: encodes with a cache
(cold, warm, full, cleared, across different texts, through the pipelined
host path) equal the encode without one, which the parity tests pin to the
oracle."""
import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _ids(tok, segs, safe):
    ids, off = tok.encode_segments(segs, tiktoken_safe=safe)
    return ids.cpu().numpy(), off.cpu().numpy()


@pytest.fixture(scope="module")
def plain_and_cached(full_table):
    import byte_level_bpe_gb300 as tk
    plain = tk.Tokenizer(full_table, workloads.SPECIALS, max_bytes=1 << 24, max_segments=8192)
    cached = tk.Tokenizer(full_table, workloads.SPECIALS, max_bytes=1 << 24, max_segments=8192)
    cached.attach_cache(64 << 20)
    yield plain, cached
    plain.close()
    cached.close()


def _serving_segs(full_table, seed, total):
    text, off = workloads.serving_batch(full_table, seed=seed, total=total, n_req=max(16, total >> 16))
    return [(text[off[i]:off[i + 1]].tobytes(), False) for i in range(len(off) - 1)]


def test_cold_then_warm(plain_and_cached, full_table, full_enc):
    from byte_level_bpe_gb300 import native
    plain, cached = plain_and_cached
    segs = _serving_segs(full_table, 31, 6 << 20)
    exp = _ids(plain, segs, False)
    got1 = _ids(cached, segs, False)
    hits1, ins1 = native.tk_last_cache_stats(cached.workspace)
    got2 = _ids(cached, segs, False)
    hits2, ins2 = native.tk_last_cache_stats(cached.workspace)
    for got in (got1, got2):
        assert np.array_equal(got[0], exp[0]) and np.array_equal(got[1], exp[1])
    assert ins1 > 0 and hits2 >= ins1 and ins2 == 0
    # sampled requests against the oracle as well
    for r in [0, 3, len(segs) - 1]:
        assert np.array_equal(got2[0][got2[1][r]:got2[1][r + 1]], full_enc.encode(segs[r][0]))


def test_other_texts_and_agentic(plain_and_cached, full_table):
    plain, cached = plain_and_cached
    for segs, safe in [(_serving_segs(full_table, 32, 3 << 20), False),
                       (workloads.agentic_segments(full_table, seed=3, scale=0.5), True),
                       (workloads.agentic_segments(full_table, seed=3, scale=0.5), True)]:
        exp = _ids(plain, segs, safe)
        got = _ids(cached, segs, safe)
        assert np.array_equal(got[0], exp[0]) and np.array_equal(got[1], exp[1])


def test_full_and_cleared_cache(full_table):
    import byte_level_bpe_gb300 as tk
    from byte_level_bpe_gb300 import native
    plain = tk.Tokenizer(full_table, workloads.SPECIALS, max_bytes=1 << 22, max_segments=4096)
    tiny = tk.Tokenizer(full_table, workloads.SPECIALS, max_bytes=1 << 22, max_segments=4096)
    cache = tiny.attach_cache(4096)  # room for a few pieces only
    segs = _serving_segs(full_table, 33, 2 << 20)
    exp = _ids(plain, segs, False)
    for _ in range(3):
        got = _ids(tiny, segs, False)
        assert np.array_equal(got[0], exp[0]) and np.array_equal(got[1], exp[1])
    n_e, n_b, n_i = native.tk_cache_stats(cache)
    assert 0 < n_b <= 4096 and n_i <= 4096
    native.tk_cache_clear(cache, torch.cuda.current_stream().cuda_stream)
    assert native.tk_cache_stats(cache) == (0, 0, 0)
    got = _ids(tiny, segs, False)
    assert native.tk_last_cache_stats(tiny.workspace)[0] == 0
    assert np.array_equal(got[0], exp[0])
    # a cache belongs to one tokenizer
    with pytest.raises(tk.TkError):
        native.tk_workspace_set_cache(plain.workspace, cache)
    plain.close()
    tiny.close()


def test_pipelined_host_call_with_cache(full_table):
    import byte_level_bpe_gb300 as tk
    segs = _serving_segs(full_table, 34, 40 << 20)
    h_text, h_off, h_allow = workloads.pack_segments(segs)
    gpu = tk.Tokenizer(full_table, workloads.SPECIALS, max_bytes=len(h_text), max_segments=len(segs))
    exp = gpu.encode_device(torch.from_numpy(h_text).cuda(), torch.from_numpy(h_off).cuda(),
                            torch.from_numpy(h_allow).cuda(), tiktoken_safe=False)
    exp = (exp[0].cpu().numpy(), exp[1].cpu().numpy())
    gpu.attach_cache(256 << 20)
    for _ in range(2):
        ids, off = gpu.encode_host(np.ascontiguousarray(h_text), h_off, h_allow, tiktoken_safe=False)
        assert np.array_equal(ids, exp[0]) and np.array_equal(off, exp[1])
    gpu.close()
