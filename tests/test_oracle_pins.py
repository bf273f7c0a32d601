"""The CPU oracle against checks that do not go through its own code (brute force, textbook LRU, closed forms,
a hand-worked trace, rejection rules)."""
import pins


def test_hand_trace():
    pins.pin_hand_trace(None)


def test_rejection_rules():
    pins.pin_rejection(None)


def test_brute_force_tiny():
    pins.pin_brute_force(None)


def test_single_selection_is_textbook_lru():
    pins.pin_textbook_lru(None)


def test_no_eviction_closed_form():
    pins.pin_no_eviction_closed_form(None)


def test_full_churn_closed_form():
    pins.pin_churn_closed_form(None)


def test_three_tier_brute_force():
    pins.pin_brute_force_tiered(None)


def test_three_tier_all_resident_closed_form():
    pins.pin_tiered_all_resident(None)
