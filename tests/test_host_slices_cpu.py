"""The slicing rule of the host entry point (no GPU): the slices tile the
batch x sequence once, in order; batch ranges are balanced; a single
sequence is cut only at chunk boundaries, never into empty segments."""
import pytest

import mamba_ssd_forward_chunked_gb300 as ssd


@pytest.mark.parametrize("batch,seqlen,q,pieces", [
    (1, 1, 64, 4), (1, 63, 64, 4), (1, 64, 64, 4), (1, 700, 128, 3), (1, 700, 128, 8), (1, 16384, 256, 4),
    (2, 2048, 256, 4), (3, 300, 128, 2), (4, 4096, 256, 4), (5, 100, 64, 3), (128, 512, 128, 4), (3, 300, 128, 1),
])
def test_slices_cover_once(batch, seqlen, q, pieces):
    sl = ssd.host_slices(batch, seqlen, q, pieces)
    assert 1 <= len(sl) <= pieces
    cover = set()
    for b0, b1, l0, l1 in sl:
        assert 0 <= b0 < b1 <= batch and 0 <= l0 < l1 <= seqlen
        for b in range(b0, b1):
            for seg in [(l0, l1)]:
                assert (b, seg) not in cover
                cover.add((b, seg))
    if batch > 1 or len(sl) == 1:
        # batch ranges over the whole sequence, contiguous, sizes differing by at most one
        assert all(l0 == 0 and l1 == seqlen for _, _, l0, l1 in sl)
        assert [s[0] for s in sl] == [0] + [s[1] for s in sl[:-1]] and sl[-1][1] == batch
        sizes = [b1 - b0 for b0, b1, _, _ in sl]
        assert max(sizes) - min(sizes) <= 1
    else:
        # one sequence: consecutive segments, each starting on a chunk boundary
        assert sl[0][2] == 0 and sl[-1][3] == seqlen
        assert all(a[3] == b[2] for a, b in zip(sl, sl[1:]))
        assert all(l0 % q == 0 for _, _, l0, _ in sl)


def test_single_chunk_is_not_split():
    assert ssd.host_slices(1, 200, 256, 4) == [(0, 1, 0, 200)]
