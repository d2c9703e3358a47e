"""CPU oracle for jagged attention -- TEST INFRASTRUCTURE ONLY (tests, smoke, bench CPU baseline)."""
