"""The host-side model of the forward kernel's barrier protocol (tests/pipeline_model.py):
every kernel variant's ring depths under random interleavings, and the model's ability to
find a real race (the D = 256 rab-ring race that a bit-exact GPU test once exposed)."""
import random

import pytest

import pipeline_model as M

CONFIGS = ([(d, rab, "epi") for d in (32, 64, 128, 256) for rab in (False, True)] +
           [(d, True, "mma") for d in (32, 64)] + [(d, True, "two") for d in (32, 64, 128)] +
           [(512, False, "epi")])


def _items(seed):
    rng = random.Random(seed)
    return [rng.randint(1, 6) for _ in range(rng.randint(1, 12))]


@pytest.mark.parametrize("d,rab,mode", CONFIGS)
def test_protocol_has_no_stale_phase_overrun_or_hang(d, rab, mode):
    """Every wait passes on exactly its phase, every buffer read finds its tile and every
    role finishes, over 400 schedules (half of them with slow loads and products), for
    every kernel variant: rab read by the epilogue, added by the tensor core, or sharing
    its ring slots with a custom mask."""
    cfg = M.kernel_cfg(d, rab, mode)
    for seed in range(200):
        for p_async in (0.5, 0.1):
            M.run(cfg, _items(seed), seed, p_async=p_async)


def test_model_finds_the_d256_rab_ring_race():
    """Without the guard (a group first waits for the other group's release of tile t - 1),
    the one-tile rab ring shared by the two D = 256 epilogue groups lets a group's parity
    wait pass on phase t - 2 for phase t: the model must report it."""
    cfg = M.kernel_cfg(256, True)
    cfg.rab_guard = False
    found = []
    for seed in range(300):
        try:
            M.run(cfg, _items(seed), seed, p_async=0.1)
        except M.Violation as e:
            found.append(str(e))
    assert found, "the unguarded rab ring raced in no schedule"
    assert any("r_full" in m for m in found), found[:3]


def test_model_finds_a_missing_free_wait():
    """A score issuer that does not wait for its S buffer to be free overwrites S(t - 2)
    before the epilogue has read it."""
    cfg = M.kernel_cfg(128, False)
    orig = M.s_issuer

    def careless(w):
        for a in orig(w):
            if a[0] == "wait" and a[1][0] == "s_free":
                continue
            yield a
    M.s_issuer = careless
    try:
        with pytest.raises(M.Violation):
            for seed in range(200):
                M.run(cfg, _items(seed), seed, p_async=0.1)
    finally:
        M.s_issuer = orig


def test_model_finds_a_tensor_core_rab_slot_released_too_early():
    """With rab added by the tensor core, a score issuer that releases the rab slot before
    its product has read it (an arrive instead of a commit behind the product) lets the
    producer overwrite the tile: the model must report the stale read."""
    cfg = M.kernel_cfg(64, True, "mma")
    orig = M.s_issuer

    def early(w):
        for a in orig(w):
            if a[0] == "commit" and a[1][0] == "r_empty":
                continue
            if a[0] == "wait" and a[1][0] == "r_full":
                yield a
                yield ("arrive", ("r_empty", a[1][1]))
                continue
            yield a
    M.s_issuer = early
    try:
        with pytest.raises(M.Violation):
            for seed in range(300):
                M.run(cfg, _items(seed), seed, p_async=0.1)
    finally:
        M.s_issuer = orig
