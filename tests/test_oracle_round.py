"""Pin of the oracle's scaffold-speculative round (composition of the pinned
attention, unmask and verify functions) on the Fast-dDrive-shaped round's
inputs: the generator plants every editable row's peak probability and makes
the AR rows agree with the draft on a seeded number k of the rows below the
threshold, then disagree; the round must commit exactly the rows at or above
the threshold, then k drafts plus the bonus token."""
import numpy as np

import oracle
import synth


def test_round_commits_threshold_rows_then_k_plus_bonus():
    inp = synth.fast_ddrive_round(synth.FAST_DDRIVE.seed)
    conf = np.asarray(inp["planted_conf"])
    assert (np.abs(conf - synth.DDRIVE_TAU) >= 1e-4).all()
    n_tau = int((conf >= synth.DDRIVE_TAU).sum())
    k = inp["planted_accept"]
    total, r, vr = oracle.speculative_round(inp["layers"][:2], inp["C"], inp["n_q"], inp["logits"],
                                            inp["logit_row"], inp["state"], inp["tokens"], inp["ar_logits"],
                                            synth.DDRIVE_TAU)
    assert int(r["n_committed"][0]) == n_tau
    assert int(vr["accepted_len"][0]) == k + 1
    assert total == n_tau + k + 1
    # every editable slot is now committed up to the bonus; the rest are masked again
    st = vr["state"][0]
    assert int((st == synth.COMMITTED).sum()) == n_tau + k + 1
