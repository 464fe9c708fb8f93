// Row reduction skeleton (written next).
