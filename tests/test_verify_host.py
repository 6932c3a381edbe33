"""Prompt-lookup drafting (host logic of the verify block), worked by hand.

Husky page, the passage before "Flash draft model and candidate selection": when
the last tokens just generated also occur in the prompt, the tokens that followed
them there are proposed (7 of them, for an 8-token verify block)."""
import pytest

from skinny_gemm_bit_gb300 import tfq as T


def draft(prompt, tail, ngram=3, k=7):
    return T.tf_draft_prompt_lookup(prompt, tail, ngram, k)


def test_the_tokens_after_the_match_are_proposed():
    assert draft([10, 11, 12, 13, 14, 15, 16, 17, 18, 19], [11, 12]) == [13, 14, 15, 16, 17, 18, 19]


def test_at_most_max_draft_tokens():
    assert draft(list(range(100, 120)), [101], k=7) == list(range(102, 109))
    assert draft(list(range(100, 120)), [101], k=2) == [102, 103]
    assert draft(list(range(100, 120)), [101], k=0) == []


def test_the_longest_suffix_wins_over_a_later_shorter_match():
    # [2, 9] occurs once, late (followed by 5, 6); [9] alone occurs first at 2
    prompt = [7, 8, 9, 1, 2, 9, 5, 6]
    assert draft(prompt, [3, 2, 9]) == [5, 6]
    assert draft(prompt, [3, 2, 9], ngram=1) == [1, 2, 9, 5, 6]  # only the last token is looked up


def test_the_first_occurrence_is_used():
    assert draft([4, 1, 2, 4, 3, 4, 6, 7], [4], ngram=1) == [1, 2, 4, 3, 4, 6, 7]
    assert draft([4, 1, 2, 4, 3, 4, 6, 7], [4], ngram=1, k=3) == [1, 2, 4]


def test_an_occurrence_with_nothing_after_it_is_skipped():
    # the prompt's own ending matches the tail but proposes nothing; the earlier one does
    assert draft([5, 6, 7, 5, 6], [5, 6]) == [7, 5, 6]
    assert draft([1, 2, 3], [2, 3]) == []


def test_no_match_gives_no_draft():
    assert draft([1, 2, 3, 4], [9, 9, 9]) == []
    assert draft([1, 2, 3, 4], []) == []


def test_bad_arguments_are_refused():
    with pytest.raises(T.TfqError):
        T.tf_draft_prompt_lookup([1, 2, 3], [1], 0, 7)  # max_ngram < 1
