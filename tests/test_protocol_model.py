"""Exhaustive check of the combine-slot protocol model (two senders, two experts, two slots,
three requests so slots are reused, cancellation at any point).  The rules mirror the device
code: pairs of a retired slot are dropped on arrival, queued ones still land, and the slot is
freed only when its last accepted result has landed."""
from oracle.slot_protocol import Model

ROUTES = [(0, 1), (1, 0), (0, 1)]


def test_protocol_safe_without_cancel():
    states, viol, dead = Model(ROUTES).explore()
    assert states > 100 and not viol and not dead


def test_protocol_safe_with_cancellation():
    for canc in [(0,), (1,), (0, 1), (0, 2), (0, 1, 2)]:
        states, viol, dead = Model(ROUTES, cancel_requests=canc).explore()
        assert not viol, (canc, viol)
        assert not dead, canc                     # every request is published or cancelled


def test_protocol_unsafe_reuse_is_caught():
    """Freeing a cancelled slot before its queued records have landed lets a late record of
    the old request land on the new owner -- the checker must find it."""
    _, viol, _ = Model(ROUTES, reuse_on_cancel=True, cancel_requests=(0,)).explore()
    kinds = {v[0] for v in viol}
    assert "foreign-write" in kinds and "mixed-output" in kinds


def test_protocol_generation_wraparound_is_harmless_under_quiescence():
    """With 1-bit generations the slot generation wraps after two reuses; the quiescence rule
    still admits no foreign write, because no record outlives its generation."""
    _, viol, dead = Model(ROUTES, cancel_requests=(0, 1), gen_bits=1).explore()
    assert not viol and not dead


def test_protocol_pool_payload_only_from_accepted_pairs():
    """The token-pool row changes only when a pair is accepted: over every interleaving (with
    cancellation, so late stale pairs exist), every record reads its own request's vector."""
    for canc in [(0,), (1,), (0, 1), (0, 1, 2)]:
        _, viol, dead = Model(ROUTES, cancel_requests=canc).explore()
        assert not viol and not dead, (canc, viol)


def test_protocol_pool_write_on_rejected_pair_is_caught():
    """Copying a rejected (stale) pair's vector into the pool row lets a late pair of a
    cancelled request replace the new owner's input before its records run -- the checker
    must find that ("foreign-input")."""
    _, viol, _ = Model(ROUTES, cancel_requests=(0,), pool_on_reject=True).explore()
    assert "foreign-input" in {v[0] for v in viol}
    _, viol, _ = Model(ROUTES, pool_on_reject=True).explore()      # without cancellation no
    assert not viol                                                  # pair is ever stale
