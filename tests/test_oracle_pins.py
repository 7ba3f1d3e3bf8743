"""The CPU oracle against facts it does not compute itself (see tests/_pins.py)."""
import pytest

import oracle
from _pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(pin):
    pin(oracle.load())


def test_oracle_rejects_bad_indices():
    import numpy as np
    from _pins import Dense
    d = Dense(91, reqs=2, G=1, H=2, B=16, RT=16)
    reg = d.regions.copy()
    reg[0, 0] = -5
    with pytest.raises(oracle.OracleError):
        d.oracle(regions=reg)
    table = d.table.copy()
    table[0, 0] = d.cache.shape[0] + 3
    with pytest.raises(oracle.OracleError):
        oracle.sparse_decode_attention(d.query, d.cache, d.regions, table, d.positions, d.active,
                                       scale=d.scale, region_tokens=d.RT)
    pos = d.positions.copy()
    pos[0] = d.table.shape[1] * d.B + 5            # visible tokens past the table width
    reg = d.regions.copy()
    reg[0, 0] = pos[0] // d.RT
    with pytest.raises(oracle.OracleError):
        d.oracle(regions=reg, positions=pos)


def test_summary_scores_rejects_bad_indices():
    import numpy as np
    from _pins import DenseSummaries
    d = DenseSummaries(5, seq_lens=[40, 20], G=2, B=16)
    d.table[0, 1] = d.summaries.shape[0]              # a page past the summary buffer
    with pytest.raises(oracle.OracleError):
        d.run(oracle.load())
    d = DenseSummaries(5, seq_lens=[40, 20], G=2, B=16)
    d.seq_lens = np.array([40 + 3 * 16, 20], np.int32)  # scored regions past the table width
    d.n_cols = 20
    with pytest.raises(oracle.OracleError):
        d.run(oracle.load())
