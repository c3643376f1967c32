"""The planted mistakes of tests/oracle_mutations.py still apply to the
oracle's source (each edited line occurs exactly once), so the mutation check
keeps testing the oracle as it stands.  The check itself is run by hand."""

import os

import oracle_mutations


def test_every_mutation_applies_to_the_current_oracle_source():
    text = open(os.path.join(oracle_mutations.ROOT, oracle_mutations.C)).read()
    assert len(oracle_mutations.M) >= 30
    for name, edits in oracle_mutations.M.items():
        for old, new in edits:
            assert old != new, name
            assert text.count(old) == 1, (name, old)
